"""The device timeline trace (cf_tuning.trace): %globaltimer stamps per CTA
(start, set-up done, role loops done, exit) and per tile (cf_trace_event /
cf_trb_event slots).  Tracing must not change a result, must write only the
grid's slots, and the stamps must respect the order the kernels impose."""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import check_softmax, dev_bf16, dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu


def _trace_buffer(torch, ctas):
    # one guard block past the grid's slots: it must stay untouched
    return torch.zeros((ctas + 1) * cf.CF_TRACE_SLOTS, dtype=torch.int64, device="cuda")


def _check_cta_stamps(T, ctas):
    T = T.view(ctas + 1, cf.CF_TRACE_SLOTS).cpu().numpy()
    assert not T[ctas].any(), "trace written past the grid's slots"
    cta = T[:ctas, :4]
    assert (cta > 0).all(), "a CTA stamp is missing"
    assert (np.diff(cta, axis=1) >= 0).all(), "CTA stamps out of order (start, set-up, loops, exit)"
    return T[:ctas, 4:].reshape(ctas, cf.CF_TRACE_TILES, cf.CF_TRACE_EVENTS)


def test_trace_fused_softmax():
    torch = torch_cuda()
    M, N, K = 512, 2048, 128
    d = inputs.gemm_inputs(M, N, K, 61, x_std=1.0, w_std=K ** -0.5, bias_std=None, gamma_std=None,
                           beta_std=None)
    st, plan, _ = cf.cf_query_gemm_fused_plan(M, N, K, 2, None)
    assert st == cf.CF_OK
    ctas = plan.clusters * plan.cluster_size * plan.cluster_m
    tr = _trace_buffer(torch, ctas)
    X, W = dev_bf16(d["X"]), dev_bf16(d["W"])
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_gemm_fused_workspace_size(M, N, K))
    cf.check(cf.cf_gemm_fused_rowsoftmax(X, W, None, Y, M, N, K, K ** -0.5, ws, ws.numel(), None,
                                         cf.tuning(trace=tr)))
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    check_softmax(host(Y), oracle.gemm_rowsoftmax(d["X"], d["W"], scale=K ** -0.5), "traced softmax",
                  bf16_out=True)
    E = _check_cta_stamps(tr, ctas)
    t0 = E[:, 0]  # every CTA's first tile
    # the MMA of a tile starts after its first operands were requested, and the
    # epilogue stores after it computed the statistics
    assert (t0[:, cf.CF_TR_MMA_FIRST] >= t0[:, cf.CF_TR_TMA_FIRST]).all()
    assert (t0[:, cf.CF_TR_EPI_STORED] >= t0[:, cf.CF_TR_EPI_STATS]).all()
    assert (t0[:, cf.CF_TR_EPI_STATS] >= t0[:, cf.CF_TR_EPI_START]).all()


@pytest.mark.parametrize("n_slice", [128, 256])
def test_trace_b2b(n_slice):
    """Stream kernel (trace tile = chunk) and cluster kernel (tile = row block)."""
    torch = torch_cuda()
    M, K, N1, N2 = 1024, 128, 1024, 128
    d = inputs.b2b_inputs(M, K, N1, N2, 62, x_std=1.0, w1_std=K ** -0.5, w2_std=1.0)
    st, plan = cf.cf_query_b2b_plan(M, K, N1, N2, cf.CF_B2B_SOFTMAX, cf.tuning(n_slice=n_slice))
    assert st == cf.CF_OK
    ctas = plan.clusters * plan.cluster_size
    tr = _trace_buffer(torch, ctas)
    X, W1, W2 = dev_bf16(d["X"]), dev_bf16(d["W1"]), dev_bf16(d["W2"])
    O = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_b2b_workspace_size())
    cf.check(cf.cf_b2b_gemm(X, W1, None, W2, O, M, K, N1, N2, K ** -0.5, cf.CF_B2B_SOFTMAX, ws, ws.numel(), None,
                            cf.tuning(n_slice=n_slice, trace=tr)))
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    ref = oracle.b2b_gemm(d["X"], d["W1"], d["W2"], op="softmax", alpha=K ** -0.5)
    o = host(O)
    assert np.abs(o - ref).max() <= 4 * 2.0 ** -8 * (np.abs(ref).max() + 1e-3)
    E = _check_cta_stamps(tr, ctas)
    t0 = E[:, 0]
    # MatMul_1 of the first tile is issued before it is committed, and the
    # epilogue sees its S after the MMA warp started it
    assert (t0[:, cf.CF_TRB_ML1_DONE] >= t0[:, cf.CF_TRB_ML1_FIRST]).all()
    assert (t0[:, cf.CF_TRB_EPI1_START] >= t0[:, cf.CF_TRB_ML1_FIRST]).all()
    assert (t0[:, cf.CF_TRB_ML2_DONE] >= t0[:, cf.CF_TRB_ML2_START]).all()


def test_trace_b2b_layernorm_stream():
    """The stream kernel's LayerNorm path (its fold kernel launched first):
    stamps in causal order and the traced result within the parity bound."""
    torch = torch_cuda()
    M, K, N1, N2 = 1024, 128, 1024, 128
    d = inputs.b2b_inputs(M, K, N1, N2, 63, x_std=1.0, w1_std=K ** -0.5, w2_std=N1 ** -0.5, b1_std=0.2, ln=True)
    st, plan = cf.cf_query_b2b_plan(M, K, N1, N2, cf.CF_B2B_LAYERNORM, cf.tuning(n_slice=128))
    assert st == cf.CF_OK and plan.cluster_size == 1
    ctas = plan.clusters
    tr = _trace_buffer(torch, ctas)
    X, W1, W2 = dev_bf16(d["X"]), dev_bf16(d["W1"]), dev_bf16(d["W2"])
    O = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_b2b_workspace_size())
    cf.check(cf.cf_b2b_gemm_layernorm(X, W1, dev_f32(d["b1"]), dev_f32(d["gamma1"]), dev_f32(d["beta1"]), W2, O, M,
                                      K, N1, N2, 1.0, 1e-5, ws, ws.numel(), None, cf.tuning(n_slice=128, trace=tr)))
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK
    ref = oracle.b2b_gemm(d["X"], d["W1"], d["W2"], op="layernorm", b1=d["b1"], gamma1=d["gamma1"],
                          beta1=d["beta1"], eps=1e-5)
    o = host(O)
    assert np.abs(o - ref).max() <= 4 * 2.0 ** -8 * (np.abs(ref).max() + 1e-3)
    E = _check_cta_stamps(tr, ctas)
    t0 = E[:, 0]
    assert (t0[:, cf.CF_TRB_ML1_DONE] >= t0[:, cf.CF_TRB_ML1_FIRST]).all()
    assert (t0[:, cf.CF_TRB_EPI1_START] >= t0[:, cf.CF_TRB_ML1_FIRST]).all()
    assert (t0[:, cf.CF_TRB_ML2_DONE] >= t0[:, cf.CF_TRB_ML2_START]).all()
