"""GPU parity of the stitched normalisation subgraphs (through the C ABI)
against the fp64 oracle: add + LayerNorm over rows (packed and split
mappings, with and without R, in place, the scalar path for ragged widths)
and BatchNorm over columns (Regional and Global schemes, ragged strips, the
batch statistics, agreement of the two schemes, repeatability, the grid
barrier's bounded wait), plus the page-shaped workloads.

Tolerance (fp32 in, fp32 out; the pages give none for these subgraphs): the
statistics are fp32 sums over at most a few thousand terms per thread
followed by a fixed tree, so the relative error of the mean and variance
stays near 1e-5 of the row or column spread; the outputs are O(1) (gamma ~ 1,
beta ~ 0.1).  Checked: max-abs <= 1e-4 + 1e-5 |ref| and mean-abs <= 1e-5.
"""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import dev_f32, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu


def check_close(y, ref, what):
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    bound = 1e-4 + 1e-5 * np.abs(ref)
    worst = np.argmax(err - bound)
    assert err.flat[worst] <= bound.flat[worst], (
        f"{what}: error {err.flat[worst]:.3e} at |ref| = {abs(ref.flat[worst]):.3f}")
    assert err.mean() <= 1e-5, f"{what}: mean-abs {err.mean():.3e}"


def _shifted(x):
    """x on the device at an address 4 bytes past a 16-byte boundary."""
    torch = torch_cuda()
    buf = torch.empty(x.size + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)))
    return buf[1:]


def _addln(d, eps=1e-5, tuning=None, in_place=False, use_R=True, params_16b=True):
    torch = torch_cuda()
    rows, cols = d["A"].shape
    A = dev_f32(d["A"])
    R = dev_f32(d["R"]) if use_R else None
    out = A if in_place else torch.full_like(A, float("nan"))
    ws = cf.new_workspace(cf.cf_stitch_workspace_size(rows, cols))
    g, b = (dev_f32(d["gamma"]), dev_f32(d["beta"])) if params_16b else (_shifted(d["gamma"]), _shifted(d["beta"]))
    st = cf.cf_stitch_add_layernorm(A, R, g, b, out, rows, cols, eps, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("rows,cols", [(1000, 32), (777, 20), (3000, 128), (513, 7), (300, 1), (64, 30000),
                                       (10, 4097), (3, 65536)])
def test_add_layernorm_shapes(rows, cols):
    d = inputs.stitch_norm_inputs(rows, cols, seed=rows + cols)
    y = _addln(d)
    ref = oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], 1e-5)
    check_close(y, ref, f"add+LN {rows}x{cols}")


@pytest.mark.parametrize("rows,cols,C,clusters,aligned", [(21, 8192, 4, 3, True), (21, 8192, 4, 3, False),
                                                        (10, 30000, 8, 2, True), (7, 4097, 2, 1, True)])
def test_add_layernorm_split_rows_per_cluster(rows, cols, C, clusters, aligned):
    """Fewer clusters than rows: each cluster walks several rows, reusing its
    exchange slots by row parity and (16-byte aligned rows) the gamma/beta it
    staged in shared memory for the first row."""
    d = inputs.stitch_norm_inputs(rows, cols, seed=rows * 7 + cols + C)
    ref = oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], 1e-5)
    t = cf.tuning(stitch_mapping=2, cluster_size=C, max_clusters=clusters)
    check_close(_addln(d, tuning=t, params_16b=aligned), ref, f"add+LN split {rows}x{cols} C={C} x{clusters}")


@pytest.mark.parametrize("rows,cols", [(1000, 32), (64, 30000), (40, 8192)])
def test_add_layernorm_params_not_16_byte_aligned(rows, cols):
    """gamma and beta 4 bytes past a 16-byte boundary: the kernels read them
    with scalar loads (the 128-bit path, and the split kernel's shared-memory
    staging of gamma and beta, need 16-byte aligned vectors)."""
    d = inputs.stitch_norm_inputs(rows, cols, seed=rows + 3 * cols)
    ref = oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], 1e-5)
    check_close(_addln(d, params_16b=False), ref, f"add+LN {rows}x{cols}, shifted gamma/beta")


@pytest.mark.parametrize("kw", [dict(stitch_mapping=2, cluster_size=2), dict(stitch_mapping=2, cluster_size=8),
                                dict(stitch_mapping=2, cluster_size=16), dict(stitch_mapping=1)])
def test_add_layernorm_mappings(kw):
    rows, cols = 150, 96
    d = inputs.stitch_norm_inputs(rows, cols, seed=5)
    y = _addln(d, tuning=cf.tuning(**kw))
    ref = oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], 1e-5)
    check_close(y, ref, f"add+LN {kw}")


def test_add_layernorm_without_residual_and_in_place():
    d = inputs.stitch_norm_inputs(900, 48, seed=6)
    ref0 = oracle.stitch_add_layernorm(d["A"], None, d["gamma"], d["beta"], 1e-5)
    check_close(_addln(d, use_R=False), ref0, "add+LN R = NULL")
    ref = oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], 1e-5)
    check_close(_addln(d, in_place=True), ref, "add+LN in place")


def test_add_layernorm_split_in_place():
    d = inputs.stitch_norm_inputs(20, 5000, seed=7)
    ref = oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], 1e-5)
    check_close(_addln(d, in_place=True), ref, "add+LN split in place")


def _bn(d, eps=1e-5, tuning=None, ws=None):
    torch = torch_cuda()
    rows, cols = d["A"].shape
    A = dev_f32(d["A"])
    out = torch.full_like(A, float("nan"))
    mean = torch.full((cols,), float("nan"), device="cuda")
    var = torch.full((cols,), float("nan"), device="cuda")
    if ws is None:
        ws = cf.new_workspace(cf.cf_stitch_batchnorm_workspace_size(rows, cols))
    st = cf.cf_stitch_batchnorm(A, dev_f32(d["gamma"]), dev_f32(d["beta"]), out, mean, var, rows, cols, eps, ws,
                                ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return (out.cpu().numpy().astype(np.float64), mean.cpu().numpy().astype(np.float64),
            var.cpu().numpy().astype(np.float64))


def _check_bn(d, got, what, eps=1e-5):
    y, m, v = got
    ref, rm, rv = oracle.stitch_batchnorm(d["A"], d["gamma"], d["beta"], eps)
    check_close(y, ref, what)
    assert np.allclose(m, rm, rtol=1e-5, atol=1e-5), f"{what}: batch mean"
    assert np.allclose(v, rv, rtol=1e-4, atol=1e-5), f"{what}: batch variance"


@pytest.mark.parametrize("rows,cols", [(64, 30000), (200, 1000), (256, 130), (1, 50), (9, 3), (100, 4096)])
def test_batchnorm_regional(rows, cols):
    d = inputs.stitch_norm_inputs(rows, cols, seed=rows * 3 + cols, with_R=False)
    st, mapping, grid = cf.cf_query_stitch_batchnorm_plan(rows, cols)
    assert st == cf.CF_OK and mapping == 3
    _check_bn(d, _bn(d), f"BN Regional {rows}x{cols}")


@pytest.mark.parametrize("rows,cols", [(5000, 36), (100000, 520), (257, 8), (20000, 1), (40000, 64),
                                       (3000, 1000)])
def test_batchnorm_global(rows, cols):
    d = inputs.stitch_norm_inputs(rows, cols, seed=rows + 7 * cols, with_R=False)
    st, mapping, grid = cf.cf_query_stitch_batchnorm_plan(rows, cols)
    assert st == cf.CF_OK and mapping == 4 and grid >= 1
    _check_bn(d, _bn(d), f"BN Global {rows}x{cols}")


@pytest.mark.parametrize("rows,cols", [(5000, 36), (100000, 520), (40000, 64), (3000, 1000)])
def test_batchnorm_global_unstreamed(rows, cols):
    """The Global scheme with plain loads (tuning stitch_mapping 5) instead of
    the TMA-streamed kernel the planner picks for 128-bit rows."""
    d = inputs.stitch_norm_inputs(rows, cols, seed=rows + 5 * cols, with_R=False)
    _check_bn(d, _bn(d, tuning=cf.tuning(stitch_mapping=5)), f"BN Global unstreamed {rows}x{cols}")


def test_batchnorm_schemes_agree_and_repeat():
    d = inputs.stitch_norm_inputs(240, 72, seed=9, with_R=False)
    a = _bn(d, tuning=cf.tuning(stitch_mapping=3))
    b = _bn(d, tuning=cf.tuning(stitch_mapping=4))
    c = _bn(d, tuning=cf.tuning(stitch_mapping=5))
    _check_bn(d, a, "BN Regional forced")
    _check_bn(d, b, "BN Global forced (TMA-streamed)")
    _check_bn(d, c, "BN Global forced (plain loads)")
    assert np.allclose(a[0], b[0], rtol=1e-5, atol=1e-5) and np.allclose(b[0], c[0], rtol=1e-5, atol=1e-5)
    d2 = inputs.stitch_norm_inputs(30000, 32, seed=10, with_R=False)
    r1, r2 = _bn(d2), _bn(d2)
    assert all(np.array_equal(x, y) for x, y in zip(r1, r2)), "Global BatchNorm not bitwise repeatable"
    u1, u2 = _bn(d2, tuning=cf.tuning(stitch_mapping=5)), _bn(d2, tuning=cf.tuning(stitch_mapping=5))
    assert all(np.array_equal(x, y) for x, y in zip(u1, u2)), "unstreamed Global BatchNorm not bitwise repeatable"
    # 32 columns make every stage one contiguous block (untiled bulk copies);
    # stitch_mapping 6 forces the tiled copies: same arithmetic, same bits
    t6 = _bn(d2, tuning=cf.tuning(stitch_mapping=6))
    assert all(np.array_equal(x, y) for x, y in zip(r1, t6)), "flat and tiled streaming differ"
    # a grid capped to a few CTAs still covers every row
    _check_bn(d2, _bn(d2, tuning=cf.tuning(max_clusters=3)), "BN Global 3 CTAs")


@pytest.mark.parametrize("rows,cols", [(200000, 32), (60000, 4), (40000, 520)])
def test_batchnorm_global_ring_and_resident_split(rows, cols):
    """The TMA-streamed Global kernel splits its stage buffers into a
    streaming ring (tuning `stages`) and stages held resident from the first
    pass to the second: every split, from a 2-stage ring with the most
    resident to no resident stage at all, gives the same bits."""
    d = inputs.stitch_norm_inputs(rows, cols, seed=rows + 11 * cols, with_R=False)
    ref = _bn(d)
    _check_bn(d, ref, f"BN Global {rows}x{cols} default split")
    for stages in (2, 3, 13, 26, 100):
        got = _bn(d, tuning=cf.tuning(stages=stages))
        assert all(np.array_equal(x, y) for x, y in zip(ref, got)), f"{rows}x{cols}: stages={stages} differs"


def test_batchnorm_grid_barrier_timeout_is_reported():
    """One arrival more than can happen: every CTA's bounded wait runs out,
    the error word says so, and the context stays usable."""
    torch = torch_cuda()
    d = inputs.stitch_norm_inputs(4000, 32, seed=11, with_R=False)
    rows, cols = d["A"].shape
    ws = cf.new_workspace(cf.cf_stitch_batchnorm_workspace_size(rows, cols))
    A = dev_f32(d["A"])
    out = torch.empty_like(A)
    st = cf.cf_stitch_batchnorm(A, dev_f32(d["gamma"]), dev_f32(d["beta"]), out, None, None, rows, cols, 1e-5, ws,
                                ws.numel(), None, cf.tuning(extra_arrivals=1, timeout_us=2000))
    assert st == cf.CF_OK
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_ERR_DEVICE_TIMEOUT and (info >> 24) == 0x72
    assert cf.cf_workspace_init(ws, ws.numel()) == cf.CF_OK
    _check_bn(d, _bn(d, ws=ws), "BN after a timeout")


def test_stitch_norm_empty_and_invalid():
    torch = torch_cuda()
    A = torch.zeros((4, 4), device="cuda")
    g = torch.ones(4, device="cuda")
    ws = cf.new_workspace(4096)
    assert cf.cf_stitch_add_layernorm(A, None, g, g, A, 0, 4, 1e-5, ws, 4096) == cf.CF_OK
    assert cf.cf_stitch_add_layernorm(A, None, g, g, A, 4, 0, 1e-5, ws, 4096) == cf.CF_OK
    assert cf.cf_stitch_add_layernorm(A, None, None, g, A, 4, 4, 1e-5, ws, 4096) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_stitch_batchnorm(A, g, g, A, None, None, 0, 4, 1e-5, ws, 4096) == cf.CF_OK
    assert cf.cf_stitch_batchnorm(A, g, g, A, None, None, -1, 4, 1e-5, ws, 4096) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_stitch_batchnorm(A, g, g, A, None, None, 1000, 4, 1e-5, ws, 256) == cf.CF_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["addln_750000x32", "addln_64x30000"])
def test_add_layernorm_workloads(name):
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(name)
    y = _addln(d, eps=w.eps)
    rows = sample_rows(w.rows, 2048, seed=3)
    ref = oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], w.eps, rows=rows)
    check_close(y[rows], ref, name)


@pytest.mark.parametrize("name", ["bn_750000x32", "bn_64x30000"])
def test_batchnorm_workloads(name):
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(name)
    _check_bn(d, _bn(d, eps=w.eps), name, eps=w.eps)
