"""GPU parity of the stitched reduce -> broadcast subgraph (through the C ABI)
against the fp64 oracle: packed and split mappings, peer and leader-follower
cluster aggregation, the 128-bit and scalar paths, ragged and empty shapes,
and the two full irregular shapes (sampled rows)."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_softmax, dev_f32, host, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu


def _run(A, b, tuning=None, out=None):
    torch = torch_cuda()
    rows, cols = A.shape
    O = out if out is not None else torch.full_like(A, float("nan"))
    ws = cf.new_workspace(cf.cf_stitch_workspace_size(rows, cols))
    st = cf.cf_stitch_rowreduce_broadcast(A, b, O, rows, cols, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    return O


@pytest.mark.parametrize("rows,cols", [(1000, 32), (777, 32), (513, 16), (100, 4), (65, 128),
                                       (31, 64), (7, 1), (9, 3), (37, 30), (50, 127)])
def test_packed_mapping(rows, cols):
    d = inputs.stitch_inputs(rows, cols, 3)
    O = _run(dev_f32(d["A"]), dev_f32(d["row_bias"]))
    check_softmax(host(O), oracle.stitch_rowreduce_broadcast(d["A"], d["row_bias"]), f"packed {rows}x{cols}")


@pytest.mark.parametrize("rows,cols,C,leader", [
    (3, 130, 1, 0), (4, 1000, 2, 0), (4, 1000, 4, 1), (2, 4097, 8, 0), (5, 30000, 8, 0),
    (5, 30000, 8, 1), (3, 30000, 16, 0), (3, 30000, 16, 1), (2, 65536, 16, 0), (6, 2050, 3, 0),
    # CTAs whose column slice is empty (their partial is (-inf, 0)), one ragged group
    (2, 70, 16, 0), (2, 70, 16, 1), (3, 66, 16, 0),
])
def test_split_mapping(rows, cols, C, leader):
    d = inputs.stitch_inputs(rows, cols, 3)
    t = cf.tuning(stitch_mapping=2, cluster_size=C, peer_max=-1 if leader else 16)
    O = _run(dev_f32(d["A"]), dev_f32(d["row_bias"]), t)
    check_softmax(host(O), oracle.stitch_rowreduce_broadcast(d["A"], d["row_bias"]),
                  f"split {rows}x{cols} C={C} leader={leader}")


@pytest.mark.parametrize("rows,cols,C,clusters,leader", [
    (9, 30000, 8, 2, 0), (17, 4100, 4, 3, 1), (40, 1000, 2, 7, 0), (5, 30000, 16, 1, 0), (33, 130, 1, 4, 0),
])
def test_split_several_rows_per_cluster(rows, cols, C, clusters, leader):
    # a cluster walks rows cid, cid + clusters, ... with the next row's loads in
    # flight while the current one is reduced, exchanged and stored; ragged row
    # counts leave some clusters one row short
    d = inputs.stitch_inputs(rows, cols, 6)
    t = cf.tuning(stitch_mapping=2, cluster_size=C, max_clusters=clusters, peer_max=-1 if leader else 16)
    O = _run(dev_f32(d["A"]), dev_f32(d["row_bias"]), t)
    check_softmax(host(O), oracle.stitch_rowreduce_broadcast(d["A"], d["row_bias"]),
                  f"split {rows}x{cols} C={C} clusters={clusters}")


def test_packed_and_split_agree():
    d = inputs.stitch_inputs(300, 128, 5)
    A, b = dev_f32(d["A"]), dev_f32(d["row_bias"])
    p = host(_run(A, b, cf.tuning(stitch_mapping=1)))
    s = host(_run(A, b, cf.tuning(stitch_mapping=2, cluster_size=2)))
    assert np.abs(p - s).max() <= 1e-5


def test_scalar_path_on_unaligned_pointers():
    torch = torch_cuda()
    d = inputs.stitch_inputs(64, 33, 3)
    rows, cols = 64, 32
    buf = torch.from_numpy(d["A"].reshape(-1)).cuda()
    A = buf[1:1 + rows * cols].view(rows, cols)  # 4-byte aligned, not 16
    assert A.data_ptr() % 16 != 0
    a_np = d["A"].reshape(-1)[1:1 + rows * cols].reshape(rows, cols)
    O = _run(A, dev_f32(d["row_bias"]))
    check_softmax(host(O), oracle.stitch_rowreduce_broadcast(a_np, d["row_bias"]), "unaligned")


def test_row_bias_is_a_shift():
    """softmax is invariant to a per-row constant: the bias must not change the result."""
    d = inputs.stitch_inputs(256, 32, 3)
    A = dev_f32(d["A"])
    o1 = host(_run(A, dev_f32(d["row_bias"])))
    o0 = host(_run(A, dev_f32(np.zeros(256, np.float32))))
    assert np.abs(o1 - o0).max() <= 1e-5


def test_empty_inputs_are_noops():
    torch = torch_cuda()
    ws = cf.new_workspace(256)
    A = torch.zeros(0, 32, device="cuda")
    assert cf.cf_stitch_rowreduce_broadcast(A, A, A, 0, 32, ws, ws.numel()) == cf.CF_OK
    assert cf.cf_stitch_rowreduce_broadcast(A, A, A, 4, 0, ws, ws.numel()) == cf.CF_OK


def test_deterministic():
    d = inputs.stitch_inputs(16, 30000, 3)
    A, b = dev_f32(d["A"]), dev_f32(d["row_bias"])
    o1 = host(_run(A, b))
    o2 = host(_run(A, b))
    assert np.array_equal(o1, o2)


@pytest.mark.parametrize("name", ["stitch_750000x32", "stitch_64x30000"])
def test_full_size_sampled(name):
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(name)
    O = _run(dev_f32(d["A"]), dev_f32(d["row_bias"]))
    rows = sample_rows(w.rows, 4096 if w.rows > 4096 else w.rows)
    ref = oracle.stitch_rowreduce_broadcast(d["A"], d["row_bias"], rows=rows)
    check_softmax(host(O)[rows], ref, name)
