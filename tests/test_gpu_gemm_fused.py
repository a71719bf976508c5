"""GPU parity of the fused GEMM + row-reduce/broadcast kernels (through the C
ABI) against the fp64 oracle: LayerNorm, GELU+LayerNorm and softmax
epilogues; ragged row tails; tile widths 64/128/256; cluster sizes 1..16;
peer and leader-follower aggregation; the global partial-buffer path; the
full workloads on every row; determinism, invariants and the device
timeout path (a bounded wait that runs out, reported without a fault)."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, check_ln_all_rows, check_softmax, dev_bf16, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


def _ln_inputs(M, N, K, seed, bias_std=0.1):
    return inputs.gemm_inputs(M, N, K, seed, x_std=K ** -0.5, w_std=K ** -0.5,
                              bias_std=bias_std, gamma_std=0.1, beta_std=0.1)


def _rownorm(d, act="none", alpha=1.0, eps=1e-5, tuning=None, bias=True, ws=None):
    torch = torch_cuda()
    X, W = dev_bf16(d["X"]), dev_bf16(d["W"])
    M, K = d["X"].shape
    N = d["W"].shape[1]
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    if ws is None:
        ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
    a = {"none": cf.CF_ACT_NONE, "gelu_tanh": cf.CF_ACT_GELU_TANH}[act]
    st = cf.cf_gemm_fused_rownorm(X, W, dev_f32(d["bias"]) if bias else None, dev_f32(d["gamma"]),
                                  dev_f32(d["beta"]), Y, M, N, K, alpha, eps, a, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return host(Y)


def _softmax(d, scale, bias=None, tuning=None):
    torch = torch_cuda()
    X, W = dev_bf16(d["X"]), dev_bf16(d["W"])
    M, K = d["X"].shape
    N = d["W"].shape[1]
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
    st = cf.cf_gemm_fused_rowsoftmax(X, W, dev_f32(bias), Y, M, N, K, scale, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return host(Y)


def _ref_ln(d, act="none", alpha=1.0, eps=1e-5, bias=True, rows=None):
    return oracle.gemm_bias_rownorm(d["X"], d["W"], d["bias"] if bias else None, d["gamma"], d["beta"],
                                    alpha=alpha, eps=eps, act=act, rows=rows)


# ---------------------------------------------------------------------------
# the tiny workload, whole
# ---------------------------------------------------------------------------
def test_ln_tiny_workload():
    w = inputs.WORKLOADS["ln_tiny_128x512x256"]
    d = inputs.workload_inputs(w.name)
    check_ln(_rownorm(d, eps=w.eps), _ref_ln(d, eps=w.eps), w.name, strict=True)


# ---------------------------------------------------------------------------
# small shapes spanning several tiles, clusters and a ragged row tail
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K,act", [
    (300, 512, 256, "none"), (300, 512, 256, "gelu_tanh"), (129, 1024, 128, "none"),
    (1, 256, 64, "none"), (257, 2048, 192, "gelu_tanh"), (640, 4096, 128, "gelu_tanh"),
])
def test_rownorm_small(M, N, K, act):
    d = _ln_inputs(M, N, K, seed=M + N + K)
    check_ln(_rownorm(d, act=act), _ref_ln(d, act=act), f"{M}x{N}x{K} {act}")


@pytest.mark.parametrize("n_slice", [64, 128, 256, 512])
def test_rownorm_tile_widths(n_slice):
    d = _ln_inputs(200, 1024, 128, seed=7)
    check_ln(_rownorm(d, tuning=cf.tuning(n_slice=n_slice)), _ref_ln(d), f"n_slice={n_slice}")


@pytest.mark.parametrize("C,leader", [(1, 0), (2, 0), (4, 0), (4, 1), (8, 0), (8, 1), (16, 0), (16, 1)])
def test_rownorm_cluster_modes(C, leader):
    """All CTAs of a row in one cluster of C; peer all-to-all or leader-follower."""
    N = 256 * C
    d = _ln_inputs(260, N, 128, seed=11 + C)
    t = cf.tuning(cluster_size=C, peer_max=-1 if leader else 16)
    check_ln(_rownorm(d, act="gelu_tanh", tuning=t), _ref_ln(d, act="gelu_tanh"), f"C={C} leader={leader}")


@pytest.mark.parametrize("C,N,leader", [(2, 2048, 0), (4, 4096, 1), (1, 1024, 0), (8, 8192, 0)])
def test_rownorm_global_path(C, N, leader):
    """Rows wider than one cluster: G = N/(256 C) clusters meet at the in-kernel barrier."""
    d = _ln_inputs(390, N, 128, seed=21 + C)
    t = cf.tuning(cluster_size=C, peer_max=-1 if leader else 16)
    check_ln(_rownorm(d, tuning=t), _ref_ln(d), f"global C={C} N={N}")


@pytest.mark.parametrize("C,CM,N,M,leader", [(1, 2, 1024, 390, 0), (2, 2, 1024, 390, 0), (4, 2, 2048, 300, 1),
                                               (8, 2, 2048, 260, 0), (2, 2, 4096, 384, 0), (1, 2, 256, 129, 0)])
def test_rownorm_pair_clusters(C, CM, N, M, leader):
    """Clusters of two row blocks x C_N column slices run CTA pairs as one cta_group::2
    MMA stream (M = 256, each CTA stages half of W); an odd row-block count leaves a
    phantom block."""
    d = _ln_inputs(M, N, 192, seed=41 + C + N)
    t = cf.tuning(cluster_size=C, cluster_m=CM, peer_max=-1 if leader else 16)
    st, plan, _ = cf.cf_query_gemm_fused_plan(M, N, 192, 1, t)
    assert st == cf.CF_OK and plan.cluster_m == CM and plan.cluster_size == C
    check_ln(_rownorm(d, act="gelu_tanh", tuning=t), _ref_ln(d, act="gelu_tanh"), f"C={C} CM={CM} N={N}")


@pytest.mark.parametrize("C,leader,epi,M,K,max_clusters", [
    (1, 0, "none", 300, 256, 0), (2, 0, "gelu_tanh", 260, 128, 0), (4, 0, "softmax", 300, 128, 0),
    (4, 1, "gelu_tanh", 200, 192, 0), (8, 0, "none", 129, 64, 0), (8, 1, "softmax", 257, 128, 0),
    (2, 0, "softmax", 1000, 128, 2), (2, 1, "gelu_tanh", 1100, 64, 1),
])
def test_wide_tile_modes(C, leader, epi, M, K, max_clusters):
    """Wide tiles (n_slice 512: all of tensor memory, both epilogue groups on one tile,
    their half-row statistics combined in shared memory) in clusters of C, peer or
    leader-follower; with few clusters every CTA runs several wide tiles in a row
    (one accumulator: phases and exchange sets advance every tile)."""
    N = 512 * C
    t = cf.tuning(n_slice=512, cluster_size=C, peer_max=-1 if leader else 16, max_clusters=max_clusters)
    kind = 2 if epi == "softmax" else (1 if epi == "gelu_tanh" else 0)
    st, plan, _ = cf.cf_query_gemm_fused_plan(M, N, K, kind, t)
    assert st == cf.CF_OK and plan.n_slice == 512 and plan.groups == 1 and plan.cluster_size == C
    if epi == "softmax":
        d = inputs.gemm_inputs(M, N, K, seed=90 + C, x_std=1.0, w_std=K ** -0.5,
                               bias_std=0.5, gamma_std=None, beta_std=None)
        ref = oracle.gemm_rowsoftmax(d["X"], d["W"], scale=K ** -0.5, bias=d["bias"])
        check_softmax(_softmax(d, K ** -0.5, bias=d["bias"], tuning=t), ref, f"wide softmax C={C}", bf16_out=True)
    else:
        d = _ln_inputs(M, N, K, seed=95 + C)
        check_ln(_rownorm(d, act=epi, tuning=t), _ref_ln(d, act=epi), f"wide {epi} C={C} leader={leader}")


def test_softmax_pair_clusters():
    d = inputs.gemm_inputs(300, 2048, 1024, seed=8, x_std=1.0, w_std=1024 ** -0.5,
                           bias_std=None, gamma_std=None, beta_std=None)
    ref = oracle.gemm_rowsoftmax(d["X"], d["W"], scale=0.05)
    for t in (cf.tuning(cluster_size=4, cluster_m=2), cf.tuning(cluster_size=8, cluster_m=2)):
        check_softmax(_softmax(d, 0.05, tuning=t), ref, "softmax CTA pairs", bf16_out=True)


def test_rownorm_alpha_and_no_bias():
    d = _ln_inputs(200, 512, 128, seed=5)
    check_ln(_rownorm(d, alpha=0.37, bias=False), _ref_ln(d, alpha=0.37, bias=False), "alpha, no bias")


def test_layernorm_invariant_on_gpu():
    """gamma=1, beta=0, eps=0: each output row has mean 0 and variance 1 (to bf16 rounding)."""
    d = _ln_inputs(256, 1024, 256, seed=9)
    d["gamma"] = np.ones(1024, np.float32)
    d["beta"] = np.zeros(1024, np.float32)
    y = _rownorm(d, act="gelu_tanh", eps=0.0)
    assert np.abs(y.mean(1)).max() < 5e-3
    assert np.abs(y.var(1) - 1).max() < 1e-2


def test_rownorm_deterministic_and_workspace_reusable():
    torch = torch_cuda()
    d = _ln_inputs(300, 2048, 128, seed=3)
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(300, 2048, 128))
    t = cf.tuning(cluster_size=2)  # global path, counters reused by every call
    ys = [_rownorm(d, tuning=t, ws=ws) for _ in range(3)]
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[1], ys[2])
    assert int(ws[256:256 + 8 * 3].sum().item()) == 0  # counters cleaned themselves
    del torch


# ---------------------------------------------------------------------------
# softmax
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(300, 2048, 128), (128, 512, 64), (77, 1024, 256)])
def test_softmax_small(M, N, K):
    d = inputs.gemm_inputs(M, N, K, seed=M + N, x_std=1.0, w_std=K ** -0.5,
                           bias_std=None, gamma_std=None, beta_std=None)
    s = K ** -0.5
    check_softmax(_softmax(d, s), oracle.gemm_rowsoftmax(d["X"], d["W"], scale=s), f"softmax {M}x{N}x{K}", bf16_out=True)


@pytest.mark.parametrize("scale,n_slice", [(128 ** -0.5, 0), (1.0, 0), (4.0, 256)])
def test_softmax_within_one_bf16_ulp(scale, n_slice):
    """Every output within one bf16 ulp of the exact value: the exponentials
    (MUFU ex2) and the row sums are fp32-accurate, so only the final rounding
    to bf16 remains.  Scale 4 gives
    peaked rows whose largest entries carry the relative error."""
    M, N, K = 300, 2048, 128
    d = inputs.gemm_inputs(M, N, K, seed=61, x_std=1.0, w_std=K ** -0.5,
                           bias_std=None, gamma_std=None, beta_std=None)
    t = cf.tuning(n_slice=n_slice) if n_slice else None
    y = _softmax(d, scale, tuning=t)
    ref = oracle.gemm_rowsoftmax(d["X"], d["W"], scale=scale)
    err = np.abs(y - ref)
    bound = np.abs(ref) * 2.0 ** -8 + 1e-30
    worst = float(np.max(err / bound))
    assert worst <= 1.0, f"scale {scale}: worst error {worst:.3f} bf16 ulps"


def test_softmax_with_bias_and_modes():
    d = inputs.gemm_inputs(200, 2048, 128, seed=4, x_std=1.0, w_std=128 ** -0.5,
                           bias_std=0.5, gamma_std=None, beta_std=None)
    ref = oracle.gemm_rowsoftmax(d["X"], d["W"], scale=0.1, bias=d["bias"])
    for t in (None, cf.tuning(peer_max=-1), cf.tuning(cluster_size=2), cf.tuning(n_slice=128)):
        check_softmax(_softmax(d, 0.1, bias=d["bias"], tuning=t), ref, f"softmax bias tuning={t}", bf16_out=True)


# ---------------------------------------------------------------------------
# the full workloads, every row against the oracle
# ---------------------------------------------------------------------------
def test_softmax_full_workload():
    w = inputs.WORKLOADS["softmax_4096x2048x128"]
    d = inputs.workload_inputs(w.name)
    y = _softmax(d, w.scale)
    check_softmax(y, oracle.gemm_rowsoftmax(d["X"], d["W"], scale=w.scale), w.name, bf16_out=True, strict=True)


@pytest.mark.parametrize("name", ["gelu_ln_16384x4096x4096", "wide_ln_8192x16384x2048"])
def test_rownorm_full_workload(name):
    """All M rows (16384 x 4096 and 8192 x 16384), compared chunk by chunk."""
    torch = torch_cuda()
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(name)
    Y = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(w.M, w.N, w.K))
    st = cf.cf_gemm_fused_rownorm(dev_bf16(d["X"]), dev_bf16(d["W"]), dev_f32(d["bias"]), dev_f32(d["gamma"]),
                                  dev_f32(d["beta"]), Y, w.M, w.N, w.K, w.alpha, w.eps,
                                  {"none": cf.CF_ACT_NONE, "gelu_tanh": cf.CF_ACT_GELU_TANH}[w.act],
                                  ws, ws.numel(), None, None)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    check_ln_all_rows(Y, lambda rows: _ref_ln(d, act=w.act, eps=w.eps, rows=rows), name, strict=True)


# ---------------------------------------------------------------------------
# device-side failure reporting without a fault
# ---------------------------------------------------------------------------
def test_global_barrier_timeout_is_reported():
    """One more arrival than can happen: the bounded wait runs out, the kernel
    records CF_ERR_DEVICE_TIMEOUT with the row block, and finishes."""
    torch = torch_cuda()
    d = _ln_inputs(256, 1024, 64, seed=2)
    M, K, N = 256, 64, 1024
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    # 256-column tiles: four per row, two clusters of two meet at the global barrier
    t = cf.tuning(n_slice=256, cluster_size=2, extra_arrivals=1, timeout_us=20000)
    st = cf.cf_gemm_fused_rownorm(dev_bf16(d["X"]), dev_bf16(d["W"]), dev_f32(d["bias"]), dev_f32(d["gamma"]),
                                  dev_f32(d["beta"]), Y, M, N, K, 1.0, 1e-5, 0, ws, ws.numel(), None, t)
    assert st == cf.CF_OK
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_ERR_DEVICE_TIMEOUT
    assert (info >> 28) == 5 and (info & 0xFFFF) in (0, 1)  # global wait of row block 0 or 1
    # the context is still usable and the error word was cleared by the read
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    cf.check(cf.cf_workspace_init(ws, ws.numel()))
    check_ln(_rownorm(d, tuning=cf.tuning(n_slice=256, cluster_size=2), ws=ws), _ref_ln(d), "after timeout")
