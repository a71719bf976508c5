"""GPU parity of the fused GEMM + bias (+ GELU) + residual + LayerNorm/RMSNorm
call (through the C ABI) against the fp64 oracle: small shapes with ragged row
tails, both norms, the schedules of the plain calls (global partials, CTA
pairs, wide tiles), R aliasing Y, the unfused composition, the argument checks
and the FFN-sized workload on sampled rows."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, dev_bf16, dev_f32, host, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed, beta=True, r_std=0.3):
    return inputs.gemm_inputs(M, N, K, seed, x_std=K ** -0.5, w_std=K ** -0.5, bias_std=0.1,
                              gamma_std=0.1, beta_std=0.1 if beta else None, resid_std=r_std)


def _run(d, act="none", norm="layer", alpha=1.0, eps=1e-5, tuning=None, unfused=False, alias=False):
    torch = torch_cuda()
    X, W, R = dev_bf16(d["X"]), dev_bf16(d["W"]), dev_bf16(d["R"])
    M, K = d["X"].shape
    N = d["W"].shape[1]
    Y = R if alias else torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    a = {"none": cf.CF_ACT_NONE, "gelu_tanh": cf.CF_ACT_GELU_TANH}[act]
    nm = {"layer": cf.CF_NORM_LAYER, "rms": cf.CF_NORM_RMS}[norm]
    beta = dev_f32(d["beta"]) if d["beta"] is not None else None
    if unfused:
        ws = cf.new_workspace(cf.cf_unfused_workspace_size(M, N, K))
        st = cf.cf_unfused_gemm_residual_norm(X, W, dev_f32(d["bias"]), R, dev_f32(d["gamma"]), beta, Y, M, N, K,
                                              alpha, eps, a, nm, ws, ws.numel(), None)
    else:
        ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
        st = cf.cf_gemm_fused_residual_norm(X, W, dev_f32(d["bias"]), R, dev_f32(d["gamma"]), beta, Y, M, N, K,
                                            alpha, eps, a, nm, ws, ws.numel(), None, tuning)
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    if not unfused:
        dst, info = cf.cf_get_device_status(ws)
        assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return host(Y)


def _ref(d, act="none", norm="layer", alpha=1.0, eps=1e-5, rows=None):
    return oracle.gemm_bias_residual_norm(d["X"], d["W"], d["bias"], d["R"], d["gamma"], d["beta"], alpha=alpha,
                                          eps=eps, act=act, norm=norm, rows=rows)


@pytest.mark.parametrize("M,N,K,act,norm", [
    (300, 512, 256, "none", "layer"), (300, 512, 256, "gelu_tanh", "rms"), (129, 1024, 128, "none", "rms"),
    (1, 256, 64, "gelu_tanh", "layer"), (257, 2048, 192, "gelu_tanh", "layer"),
])
def test_residual_small(M, N, K, act, norm):
    d = _inputs(M, N, K, seed=M + N + K + 11, beta=(norm == "layer"))
    check_ln(_run(d, act=act, norm=norm), _ref(d, act=act, norm=norm), f"residual {M}x{N}x{K} {act} {norm}")


@pytest.mark.parametrize("kw", [dict(n_slice=512), dict(n_slice=256, cluster_size=2),
                                dict(cluster_size=2, cluster_m=2), dict(cluster_size=16, peer_max=-1)])
def test_residual_schedules(kw):
    d = _inputs(390, 4096, 128, seed=81)
    check_ln(_run(d, act="gelu_tanh", tuning=cf.tuning(**kw)), _ref(d, act="gelu_tanh"), f"residual {kw}")


def test_residual_in_place_output():
    """R and Y may be one buffer: every element is read before it is overwritten."""
    d = _inputs(300, 2048, 128, seed=82)
    check_ln(_run(d, norm="rms", alias=True), _ref(d, norm="rms"), "residual R is Y")


def test_residual_unfused_composition():
    d = _inputs(260, 2048, 128, seed=83)
    check_ln(_run(d, act="gelu_tanh", unfused=True), _ref(d, act="gelu_tanh"), "residual unfused")


def test_residual_argument_checks():
    torch = torch_cuda()
    buf = torch.zeros(1 << 16, dtype=torch.float32, device="cuda")
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(128, 256, 64))
    # no residual, R aliasing X, an unknown norm
    assert cf.cf_gemm_fused_residual_norm(buf, buf[4096:], None, None, buf, buf, buf[8192:], 128, 256, 64, 1.0,
                                          1e-5, 0, 0, ws, ws.numel()) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_gemm_fused_residual_norm(buf, buf[4096:], None, buf, buf, buf, buf[8192:], 128, 256, 64, 1.0,
                                          1e-5, 0, 0, ws, ws.numel()) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_gemm_fused_residual_norm(buf, buf[4096:], None, buf[12288:], buf, buf, buf[8192:], 128, 256, 64,
                                          1.0, 1e-5, 0, 7, ws, ws.numel()) == cf.CF_ERR_INVALID_ARG


def test_residual_full_workload():
    w = inputs.WORKLOADS["residual_ln_16384x4096x4096"]
    d = inputs.workload_inputs(w.name)
    y = _run(d, act=w.act, alpha=w.alpha, eps=w.eps)
    rows = sample_rows(w.M, 512, seed=6)
    check_ln(y[rows], _ref(d, act=w.act, alpha=w.alpha, eps=w.eps, rows=rows), w.name, strict=True)
