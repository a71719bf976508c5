"""Neighbouring kernels under programmatic dependent launch and CUDA graphs
(sass2mlir, "PDL" and the CUDA-graph sections): a chain of fused calls on one
stream in which every call consumes its predecessor's output --

    Y1 = LayerNorm(X . W1 + b) (bf16)        fused GEMM + LayerNorm
    Y2 = softmax(Y1 . W2 / sqrt(N1)) (bf16)  fused GEMM + softmax
    O  = bf16(GELU(Y2 . W3)) . W4            back-to-back GEMM
    O2 = bf16(LayerNorm(O . W5)) . W6        back-to-back GEMM, LayerNorm F
                                             (stream kernel: a fold kernel,
                                             then the GEMMs, which read O
                                             before waiting on the fold)

-- run with PDL off, with PDL on, and replayed from a captured CUDA graph
(PDL edges inside the graph).  Every kernel waits on griddepcontrol before
its first global read, so all three runs must produce the same bits; the
first stage is also checked against the oracle (its own parity tests cover
the rest)."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_ln, dev_bf16, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu

M, K, N1, N2, NB1, NB2 = 1024, 256, 512, 256, 512, 128


def _setup():
    torch = torch_cuda()
    d = inputs.gemm_inputs(M, N1, K, 41, x_std=1.0, w_std=K ** -0.5, bias_std=0.1, gamma_std=0.1, beta_std=0.1)
    rng = np.random.Generator(np.random.PCG64(42))
    W2 = inputs.round_to_bf16(rng.standard_normal((N1, N2)).astype(np.float32) * N1 ** -0.5)
    W3 = inputs.round_to_bf16(rng.standard_normal((N2, NB1)).astype(np.float32) * 4.0)
    W4 = inputs.round_to_bf16(rng.standard_normal((NB1, NB2)).astype(np.float32) * NB1 ** -0.5)
    W5 = inputs.round_to_bf16(rng.standard_normal((NB2, NB1)).astype(np.float32) * NB2 ** -0.5)
    W6 = inputs.round_to_bf16(rng.standard_normal((NB1, NB2)).astype(np.float32) * NB1 ** -0.5)
    g5 = (1.0 + 0.1 * rng.standard_normal(NB1)).astype(np.float32)
    be5 = (0.1 * rng.standard_normal(NB1)).astype(np.float32)
    t = dict(X=dev_bf16(d["X"]), W1=dev_bf16(d["W"]), b=dev_f32(d["bias"]), g=dev_f32(d["gamma"]),
             be=dev_f32(d["beta"]), W2=dev_bf16(W2), W3=dev_bf16(W3), W4=dev_bf16(W4), W5=dev_bf16(W5),
             W6=dev_bf16(W6), g5=dev_f32(g5), be5=dev_f32(be5))
    t["Y1"] = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    t["Y2"] = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    t["O"] = torch.empty((M, NB2), dtype=torch.bfloat16, device="cuda")
    t["O2"] = torch.empty((M, NB2), dtype=torch.bfloat16, device="cuda")
    t["ws1"] = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N1, K))
    t["ws2"] = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N2, N1))
    t["ws3"] = cf.new_workspace(cf.cf_b2b_workspace_size())
    t["ws4"] = cf.new_workspace(cf.cf_b2b_workspace_size())
    return torch, d, t


def _chain(t, tuning, stream=None):
    cf.check(cf.cf_gemm_fused_rownorm(t["X"], t["W1"], t["b"], t["g"], t["be"], t["Y1"], M, N1, K, 1.0, 1e-5,
                                      cf.CF_ACT_NONE, t["ws1"], t["ws1"].numel(), stream, tuning), "stage 1")
    cf.check(cf.cf_gemm_fused_rowsoftmax(t["Y1"], t["W2"], None, t["Y2"], M, N2, N1, N1 ** -0.5, t["ws2"],
                                         t["ws2"].numel(), stream, tuning), "stage 2")
    cf.check(cf.cf_b2b_gemm(t["Y2"], t["W3"], None, t["W4"], t["O"], M, N2, NB1, NB2, 1.0, cf.CF_B2B_GELU_TANH,
                            t["ws3"], t["ws3"].numel(), stream, tuning), "stage 3")
    cf.check(cf.cf_b2b_gemm_layernorm(t["O"], t["W5"], None, t["g5"], t["be5"], t["W6"], t["O2"], M, NB2, NB1, NB2,
                                      1.0, 1e-5, t["ws4"], t["ws4"].numel(), stream, tuning), "stage 4")


def _outputs(torch, t):
    torch.cuda.synchronize()
    for k in ("ws1", "ws2", "ws3", "ws4"):
        st, info = cf.cf_get_device_status(t[k])
        assert st == cf.CF_OK, (k, cf.status_string(st), hex(info))
    return [t[k].clone() for k in ("Y1", "Y2", "O", "O2")]


def _clear(t):
    for k in ("Y1", "Y2", "O", "O2"):
        t[k].fill_(float("nan"))


def test_chain_same_bits_with_pdl_and_graph():
    torch, d, t = _setup()
    _chain(t, cf.tuning(disable_pdl=1))
    ref = _outputs(torch, t)
    assert all(bool(torch.isfinite(x.float()).all()) for x in ref)
    check_ln(host(ref[0]), oracle.gemm_bias_rownorm(d["X"], d["W"], d["bias"], d["gamma"], d["beta"], eps=1e-5),
             "chain stage 1")
    for rep in range(3):
        _clear(t)
        _chain(t, None)
        got = _outputs(torch, t)
        for a, b, name in zip(ref, got, ("Y1", "Y2", "O", "O2")):
            assert torch.equal(a, b), f"PDL run {rep}: {name} differs"
    # the whole chain captured as one graph (PDL edges between its kernels)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _chain(t, None, s)
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(3):
        _clear(t)
        g.replay()
        got = _outputs(torch, t)
        for a, b, name in zip(ref, got, ("Y1", "Y2", "O", "O2")):
            assert torch.equal(a, b), f"graph replay {rep}: {name} differs"
