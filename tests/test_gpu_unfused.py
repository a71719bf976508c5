"""GPU parity of the unfused two-kernel composition (GEMM -> fp32 P -> row
kernel), the baseline the fused kernel is measured against: it must give the
oracle's result within the same tolerances, and agree with the fused call."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, check_softmax, dev_bf16, dev_f32, host, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu


def _unfused_ln(d, act):
    torch = torch_cuda()
    M, K = d["X"].shape
    N = d["W"].shape[1]
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cf.cf_unfused_workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    a = {"none": cf.CF_ACT_NONE, "gelu_tanh": cf.CF_ACT_GELU_TANH}[act]
    st = cf.cf_unfused_gemm_rownorm(dev_bf16(d["X"]), dev_bf16(d["W"]), dev_f32(d["bias"]), dev_f32(d["gamma"]),
                                    dev_f32(d["beta"]), Y, M, N, K, 1.0, 1e-5, a, ws, ws.numel())
    assert st == cf.CF_OK, cf.status_string(st)
    torch.cuda.synchronize()
    return host(Y)


@pytest.mark.parametrize("M,N,K,act", [(300, 512, 256, "none"), (257, 2048, 192, "gelu_tanh"),
                                       (129, 16384, 64, "none"), (64, 320, 640, "gelu_tanh")])
def test_unfused_rownorm(M, N, K, act):
    d = inputs.gemm_inputs(M, N, K, M + N, x_std=K ** -0.5, w_std=K ** -0.5, bias_std=0.1, gamma_std=0.1,
                           beta_std=0.1)
    ref = oracle.gemm_bias_rownorm(d["X"], d["W"], d["bias"], d["gamma"], d["beta"], act=act)
    check_ln(_unfused_ln(d, act), ref, f"unfused {M}x{N}x{K} {act}")


def test_unfused_softmax_full_workload():
    torch = torch_cuda()
    w = inputs.WORKLOADS["softmax_4096x2048x128"]
    d = inputs.workload_inputs(w.name)
    Y = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cf.cf_unfused_workspace_size(w.M, w.N, w.K), dtype=torch.uint8, device="cuda")
    st = cf.cf_unfused_gemm_rowsoftmax(dev_bf16(d["X"]), dev_bf16(d["W"]), None, Y, w.M, w.N, w.K, w.scale,
                                       ws, ws.numel())
    assert st == cf.CF_OK
    torch.cuda.synchronize()
    y = host(Y)
    rows = sample_rows(w.M, 512)
    check_softmax(y[rows], oracle.gemm_rowsoftmax(d["X"], d["W"], scale=w.scale, rows=rows), "unfused softmax",
                  bf16_out=True, strict=True)
    fused = cf.gemm_fused_rowsoftmax(dev_bf16(d["X"]), dev_bf16(d["W"]), scale=w.scale)
    assert np.abs(host(fused) - y).max() <= 1e-3


def test_unfused_rejects_too_wide_rows():
    torch = torch_cuda()
    buf = torch.empty(1024, dtype=torch.float32, device="cuda")
    assert cf.cf_unfused_gemm_rowsoftmax(buf, buf, None, buf, 128, 32768, 64, 1.0, buf, 1 << 40) == \
        cf.CF_ERR_UNSUPPORTED
