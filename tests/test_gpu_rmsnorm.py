"""GPU parity of the fused GEMM + bias (+ GELU) + RMSNorm call (through the C
ABI) against the fp64 oracle: small shapes with ragged row tails, with and
without beta and bias, every schedule the LayerNorm call has (clusters of 1 to
16, peer and leader aggregation, rows over several clusters through the global
partial buffer, CTA pairs, wide tiles), the unfused composition, and the
FFN-sized workload on sampled rows."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, dev_bf16, dev_f32, host, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed, beta=True):
    return inputs.gemm_inputs(M, N, K, seed, x_std=K ** -0.5, w_std=K ** -0.5, bias_std=0.1,
                              gamma_std=0.1, beta_std=0.1 if beta else None)


def _rms(d, act="none", alpha=1.0, eps=1e-5, tuning=None, unfused=False):
    torch = torch_cuda()
    X, W = dev_bf16(d["X"]), dev_bf16(d["W"])
    M, K = d["X"].shape
    N = d["W"].shape[1]
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a = {"none": cf.CF_ACT_NONE, "gelu_tanh": cf.CF_ACT_GELU_TANH}[act]
    beta = dev_f32(d["beta"]) if d["beta"] is not None else None
    if unfused:
        ws = cf.new_workspace(cf.cf_unfused_workspace_size(M, N, K))
        st = cf.cf_unfused_gemm_rmsnorm(X, W, dev_f32(d["bias"]), dev_f32(d["gamma"]), beta, Y, M, N, K, alpha,
                                        eps, a, ws, ws.numel(), None)
    else:
        ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
        st = cf.cf_gemm_fused_rmsnorm(X, W, dev_f32(d["bias"]), dev_f32(d["gamma"]), beta, Y, M, N, K, alpha, eps,
                                      a, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    if not unfused:
        dst, info = cf.cf_get_device_status(ws)
        assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return host(Y)


def _ref(d, act="none", alpha=1.0, eps=1e-5, rows=None):
    return oracle.gemm_bias_rmsnorm(d["X"], d["W"], d["bias"], d["gamma"], d["beta"], alpha=alpha, eps=eps,
                                    act=act, rows=rows)


@pytest.mark.parametrize("M,N,K,act,beta", [
    (300, 512, 256, "none", True), (300, 512, 256, "gelu_tanh", False), (129, 1024, 128, "none", False),
    (1, 256, 64, "none", True), (257, 2048, 192, "gelu_tanh", True),
])
def test_rmsnorm_small(M, N, K, act, beta):
    d = _inputs(M, N, K, seed=M + N + K + 3, beta=beta)
    check_ln(_rms(d, act=act), _ref(d, act=act), f"rms {M}x{N}x{K} {act} beta={beta}")


@pytest.mark.parametrize("kw", [
    dict(n_slice=64), dict(n_slice=512), dict(cluster_size=16, peer_max=-1), dict(cluster_size=8, peer_max=16),
    dict(n_slice=256, cluster_size=2), dict(cluster_size=2, cluster_m=2), dict(cluster_size=4),
])
def test_rmsnorm_schedules(kw):
    """Cluster sizes, leader/peer, global partials (n_slice 256 in clusters of 2 over
    4096 columns: 8 groups), CTA pairs, wide tiles."""
    N = 4096
    d = _inputs(390, N, 128, seed=71, beta=False)
    t = cf.tuning(**kw)
    check_ln(_rms(d, act="gelu_tanh", tuning=t), _ref(d, act="gelu_tanh"), f"rms {kw}")


def test_rmsnorm_alpha_and_eps():
    d = _inputs(200, 1024, 128, seed=73)
    check_ln(_rms(d, alpha=0.37, eps=1e-3), _ref(d, alpha=0.37, eps=1e-3), "rms alpha eps")


def test_rmsnorm_unfused_composition():
    d = _inputs(260, 2048, 128, seed=74, beta=False)
    check_ln(_rms(d, act="gelu_tanh", unfused=True), _ref(d, act="gelu_tanh"), "rms unfused")


def test_rmsnorm_full_workload():
    w = inputs.WORKLOADS["rms_16384x4096x4096"]
    d = inputs.workload_inputs(w.name)
    y = _rms(d, act=w.act, alpha=w.alpha, eps=w.eps)
    rows = sample_rows(w.M, 512, seed=5)
    check_ln(y[rows], _ref(d, act=w.act, alpha=w.alpha, eps=w.eps, rows=rows), w.name, strict=True)
