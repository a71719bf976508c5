"""GPU parity of the stitched power -> broadcast -> add -> row softmax subgraph
(through the C ABI) against the fp64 oracle: the packed and split mappings,
peer and leader-follower aggregation, clusters walking several rows (the
column powers computed once per CTA and reused by every row it handles), the
scalar path, exponents 0 and 1, and the two irregular page shapes."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_softmax, dev_f32, host, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu


def _run(A, w, p, tuning=None):
    torch = torch_cuda()
    rows, cols = A.shape
    O = torch.full_like(A, float("nan"))
    ws = cf.new_workspace(cf.cf_stitch_workspace_size(rows, cols))
    st = cf.cf_stitch_powadd_softmax(A, w, p, O, rows, cols, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    return host(O)


def _check(rows, cols, p, tuning=None, seed=21):
    d = inputs.powadd_inputs(rows, cols, seed)
    y = _run(dev_f32(d["A"]), dev_f32(d["w"]), p, tuning)
    check_softmax(y, oracle.stitch_powadd_softmax(d["A"], d["w"], p), f"powadd {rows}x{cols} p={p} {tuning}")


@pytest.mark.parametrize("rows,cols", [(1000, 32), (777, 32), (513, 16), (65, 128), (9, 3), (37, 30), (100, 4)])
def test_packed(rows, cols):
    _check(rows, cols, 2.5)


@pytest.mark.parametrize("rows,cols,C,leader", [(5, 30000, 8, 0), (3, 4097, 16, 1), (4, 1000, 2, 0), (2, 130, 1, 0)])
def test_split(rows, cols, C, leader):
    _check(rows, cols, 2.5, cf.tuning(stitch_mapping=2, cluster_size=C, peer_max=-1 if leader else 16))


@pytest.mark.parametrize("rows,cols,C,clusters", [(9, 30000, 8, 2), (40, 1000, 2, 7)])
def test_split_rows_share_the_powers(rows, cols, C, clusters):
    """A cluster walks several rows; its CTAs compute their columns' powers once."""
    _check(rows, cols, 1.7, cf.tuning(stitch_mapping=2, cluster_size=C, max_clusters=clusters))


@pytest.mark.parametrize("p", [0.0, 1.0, -1.5, 3.0])
def test_exponents(p):
    """p = 0 is the plain row softmax of A, p = 1 adds w itself, negative and
    integer exponents take the same path."""
    _check(300, 32, p)
    _check(3, 8192, p)


def test_scalar_path_on_unaligned_pointers():
    torch = torch_cuda()
    d = inputs.powadd_inputs(64, 33, 4)
    rows, cols = 64, 32
    buf = torch.from_numpy(d["A"].reshape(-1)).cuda()
    A = buf[1:1 + rows * cols].view(rows, cols)
    assert A.data_ptr() % 16 != 0
    a_np = d["A"].reshape(-1)[1:1 + rows * cols].reshape(rows, cols)
    y = _run(A, dev_f32(d["w"][:cols]), 2.5)
    check_softmax(y, oracle.stitch_powadd_softmax(a_np, d["w"][:cols], 2.5), "powadd unaligned")


def test_full_size_64x30000_every_row():
    w = inputs.WORKLOADS["powsm_64x30000"]
    d = inputs.workload_inputs(w.name)
    y = _run(dev_f32(d["A"]), dev_f32(d["w"]), w.p)
    check_softmax(y, oracle.stitch_powadd_softmax(d["A"], d["w"], w.p), w.name)


def test_full_size_750000x32_sampled():
    w = inputs.WORKLOADS["powsm_750000x32"]
    d = inputs.workload_inputs(w.name)
    y = _run(dev_f32(d["A"]), dev_f32(d["w"]), w.p)
    rows = sample_rows(w.rows, 4096)
    check_softmax(y[rows], oracle.stitch_powadd_softmax(d["A"], d["w"], w.p, rows=rows), w.name)
