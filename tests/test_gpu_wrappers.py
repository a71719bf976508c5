"""The torch-level convenience wrappers of memory_fusion_gb300.cf (allocate the
output and workspace, marshal, check the status) on small cases, each against
the fp64 oracle: a user's first call into every kernel family."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, check_softmax, dev_bf16, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


def test_gemm_wrappers():
    torch_cuda()
    M, N, K = 300, 1024, 256
    d = inputs.gemm_inputs(M, N, K, 51, x_std=1.0, w_std=K ** -0.5, resid_std=0.5)
    X, W, R = dev_bf16(d["X"]), dev_bf16(d["W"]), dev_bf16(d["R"])
    b, g, be = dev_f32(d["bias"]), dev_f32(d["gamma"]), dev_f32(d["beta"])
    y = host(cf.gemm_fused_rownorm(X, W, b, g, be, act="gelu_tanh"))
    check_ln(y, oracle.gemm_bias_rownorm(d["X"], d["W"], d["bias"], d["gamma"], d["beta"], act="gelu_tanh"),
             "rownorm wrapper")
    y = host(cf.gemm_fused_rmsnorm(X, W, b, g))
    check_ln(y, oracle.gemm_bias_rmsnorm(d["X"], d["W"], d["bias"], d["gamma"]), "rmsnorm wrapper")
    y = host(cf.gemm_fused_residual_norm(X, W, b, R, g, be, norm="layer"))
    check_ln(y, oracle.gemm_bias_residual_norm(d["X"], d["W"], d["bias"], d["R"], d["gamma"], d["beta"],
                                               norm="layer"), "residual wrapper")
    y = host(cf.gemm_fused_rowsoftmax(X, W, b, scale=0.5))
    check_softmax(y, oracle.gemm_rowsoftmax(d["X"], d["W"], scale=0.5, bias=d["bias"]), "softmax wrapper",
                  bf16_out=True)
    y = host(cf.gemm_fused_rowsoftmax_causal(X, W, scale=0.5, offset=100))
    ref = oracle.gemm_rowsoftmax_causal(d["X"], d["W"], scale=0.5, offset=100)
    check_softmax(y, ref, "causal wrapper", bf16_out=True)


def test_stitched_wrappers():
    torch = torch_cuda()
    d = inputs.stitch_inputs(500, 48, 3)
    o = cf.stitch_rowreduce_broadcast(dev_f32(d["A"]), dev_f32(d["row_bias"])).cpu().numpy()
    check_softmax(o.astype(np.float64), oracle.stitch_rowreduce_broadcast(d["A"], d["row_bias"]), "stitch wrapper")
    d = inputs.stitch_norm_inputs(700, 40, 4)
    A, R, g, be = (dev_f32(d[k]) for k in ("A", "R", "gamma", "beta"))
    o = cf.stitch_add_layernorm(A, R, g, be).cpu().numpy()
    assert np.abs(o - oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], 1e-5)).max() <= 1e-4
    o, m, v = cf.stitch_batchnorm(A, g, be)
    ref, rm, rv = oracle.stitch_batchnorm(d["A"], d["gamma"], d["beta"], 1e-5)
    assert np.abs(o.cpu().numpy() - ref).max() <= 1e-4
    assert np.allclose(m.cpu().numpy(), rm, atol=1e-5) and np.allclose(v.cpu().numpy(), rv, rtol=1e-4, atol=1e-5)
    torch.cuda.synchronize()


@pytest.mark.parametrize("op", ["softmax", "gelu_tanh", "layernorm"])
def test_b2b_wrapper(op):
    torch_cuda()
    d = inputs.b2b_inputs(200, 128, 512, 64, 52, x_std=1.0, w1_std=128 ** -0.5, w2_std=512 ** -0.5, b1_std=0.1,
                          ln=op == "layernorm")
    X, W1, W2 = dev_bf16(d["X"]), dev_bf16(d["W1"]), dev_bf16(d["W2"])
    kw = dict(gamma1=dev_f32(d["gamma1"]), beta1=dev_f32(d["beta1"])) if op == "layernorm" else {}
    o = host(cf.b2b_gemm(X, W1, W2, dev_f32(d["b1"]), op=op, alpha=0.5, **kw))
    ref = oracle.b2b_gemm(d["X"], d["W1"], d["W2"], op=op, alpha=0.5, b1=d["b1"], gamma1=d["gamma1"],
                          beta1=d["beta1"])
    # loose (the full derivation is in test_gpu_b2b): a few bf16 ulps of the output scale
    assert np.abs(o - ref).max() <= 4 * 2.0 ** -8 * (np.abs(ref).max() + 1e-3), op
