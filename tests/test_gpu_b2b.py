"""GPU parity of the back-to-back GEMM O = bf16(F(alpha X.W1 + b1)) . W2
(through the C ABI) against the fp64 oracle, on both kernels -- the cluster
kernel (N1 partitioned over C = N1/256 CTAs, tuning n_slice = 256) and the
stream kernel (one CTA per row block, N1 in 256-column chunks, n_slice = 128):
the softmax, GELU and LayerNorm epilogues, every cluster
width N1/256 in {1, 2, 4, 8} and wider N1 on the stream kernel, both output
widths, ragged rows and a ragged last K block, X resident and streamed, the
online softmax's rescaling, several row blocks per CTA or cluster (the ring,
tensor memory and exchange buffers reused across tiles), ring depths, a
selector W2 that reads S back column by column, unsupported shapes, and the
page-sized workloads on sampled rows.

Tolerance.  The kernel rounds its fp32 S to bf16 and the oracle rounds its
fp64 S to bf16; the two roundings can land one bf16 ulp apart, and the
kernel's S carries its own fp32 error e_j.  So per output element

    |O - O_ref| <= sum_j (2^-7 |s_j| + e_j) |W2_jk| + N1 2^-24 sum_j |s_j W2_jk|
                   + half a bf16 ulp of the output,

with e_j <= 2^-16 |s_j| (exp2/FMA chain); for GELU, e_j also carries the
tanh.approx absolute error 2^-10.98 times 0.5 |z_j|; for LayerNorm, the fp32
row statistics add up to 2^-14 (|s_j| + 1) (the normalised values are O(1)).  The bound assumes every
S element flips, so the mean error is checked as well: at most half a bf16
ulp of the output on average plus 2^-12 of the flip term (a flip fraction
far above what rounding noise produces fails it).

The stream kernel's softmax rounds the unnormalised exponentials to bf16 and
divides by the row sum on the fp32 output; the oracle rounds the normalised
values.  Each is a bf16 rounding of S up to a positive per-row factor, so an
element still differs by at most 2^-8 |s_j| (inside the flip term), but the
two roundings are now independent: their difference adds noise of RMS at
most 2^-9 sqrt(2/3) sqrt(sum_j s_j^2 W2_jk^2) to each output, which the mean
check allows for on that kernel.

The stream kernel's LayerNorm feeds MatMul_2 the bf16 values
t_j / rstd = (z_j - mu0) gamma1_j, mu0 the mean of the row's first 256
columns, and applies rstd, the mean correction -(mu - mu0) rstd gamma1^T W2
and beta1^T W2 to the fp32 output.  Its rounding is relative to
|t_j| = |(z_j - mu0) gamma1_j rstd| instead of |s_j|, and independent of the
oracle's: the flip term gains 2^-8 sum_j |t_j||W2_jk| and the mean check the
noise 2^-9 sqrt(2/3) sqrt(sum_j t_j^2 W2_jk^2).
"""
import numpy as np
import pytest

import oracle
from memory_fusion_gb300 import cf, inputs
from tests.gpu_util import bf16_half_ulp, dev_bf16, dev_f32, host, sample_rows, torch_cuda

pytestmark = pytest.mark.gpu

OPS = {"softmax": cf.CF_B2B_SOFTMAX, "gelu_tanh": cf.CF_B2B_GELU_TANH, "layernorm": cf.CF_B2B_LAYERNORM}


def _tuning(mode, N1, **kw):
    """cf_tuning selecting the kernel: the cluster kernel (C = N1/256 CTAs of
    256 columns) or the stream kernel (one CTA per row block, 128-column chunks)."""
    return cf.tuning(n_slice=128 if mode == "stream" else 256, **kw)


def _modes(op):
    return ["cluster", "stream"]


CASES = [(op, mode) for op in OPS for mode in _modes(op)]


def _run(d, op, alpha, tuning=None, expect=cf.CF_OK):
    torch = torch_cuda()
    M, K = d["X"].shape
    N1 = d["W1"].shape[1]
    N2 = d["W2"].shape[1]
    X, W1, W2 = dev_bf16(d["X"]), dev_bf16(d["W1"]), dev_bf16(d["W2"])
    b1 = dev_f32(d.get("b1"))
    O = torch.full((max(M, 1), N2), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_b2b_workspace_size())
    if op == "layernorm":
        st = cf.cf_b2b_gemm_layernorm(X, W1, b1, dev_f32(d["gamma1"]), dev_f32(d["beta1"]), W2, O, M, K, N1, N2,
                                      alpha, 1e-5, ws, ws.numel(), None, tuning)
    else:
        st = cf.cf_b2b_gemm(X, W1, b1, W2, O, M, K, N1, N2, alpha, OPS[op], ws, ws.numel(), None, tuning)
    assert st == expect, cf.status_string(st)
    torch.cuda.synchronize()
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_OK, (cf.status_string(dst), hex(info))
    return host(O)[:M]


def _s(d, op, z):
    if op == "softmax":
        return oracle.softmax_rows(z)
    if op == "gelu_tanh":
        return oracle.gelu_tanh(z)
    return oracle.layernorm_rows(z, d["gamma1"], d["beta1"], 1e-5)


def _shifted(d, z):
    """The stream kernel's LayerNorm operand of MatMul_2 in units of S:
    t_j = (z_j - mu0) gamma1_j rstd, mu0 the mean of the row's first 256 columns."""
    mu0 = z[:, :256].mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(z.var(axis=1, keepdims=True) + 1e-5)
    return (z - mu0) * np.asarray(d["gamma1"], np.float64) * rstd


def _terms(d, op, alpha, rows=None, mode="cluster"):
    """Per element of the output: sum_j |s_j||W2_jk|, sum_j |z_j||W2_jk|,
    sqrt(sum_j r_j^2 W2_jk^2) and sum_j |r_j||W2_jk|, r the values the kernel
    rounds to bf16 (s, or t for the stream kernel's LayerNorm)."""
    X = d["X"] if rows is None else d["X"][rows]
    z = alpha * oracle.gemm(X, d["W1"]) + (0.0 if d.get("b1") is None else np.asarray(d["b1"], np.float64))
    s = _s(d, op, z)
    r = _shifted(d, z) if (op == "layernorm" and mode == "stream") else s
    aw = np.abs(np.asarray(d["W2"], np.float64))
    return np.abs(s) @ aw, np.abs(z) @ aw, np.sqrt((r * r) @ (aw * aw)), np.abs(r) @ aw


def check_b2b(o, ref, d, op, alpha, what, rows=None, mode="cluster"):
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    N1 = d["W1"].shape[1]
    A, Z, Q, R = _terms(d, op, alpha, rows, mode)
    flip = (2.0 ** -7 + 2.0 ** -16 + N1 * 2.0 ** -24) * A
    if op == "gelu_tanh":
        flip = flip + 0.5 * 2.0 ** -10.98 * Z
    if op == "layernorm":  # fp32 statistics: an error near 2^-14 of the row spread in each S element
        flip = flip + 2.0 ** -14 * (A + np.abs(np.asarray(d["W2"], np.float64)).sum(axis=0))
        if mode == "stream":
            flip = flip + 2.0 ** -8 * R
    bound = flip + bf16_half_ulp(np.abs(ref) + flip)
    err = np.abs(o - ref)
    worst = np.argmax(err - bound)
    assert err.flat[worst] <= bound.flat[worst], (
        f"{what}: error {err.flat[worst]:.3e} > bound {bound.flat[worst]:.3e} at |ref|={abs(ref.flat[worst]):.3e}")
    mean_bound = bf16_half_ulp(np.abs(ref)).mean() + 2.0 ** -12 * flip.mean()
    if mode == "stream" and op in ("softmax", "layernorm"):  # independent roundings (module docstring)
        mean_bound += 2.0 ** -9 * np.sqrt(2.0 / 3.0) * Q.mean()
    assert err.mean() <= mean_bound, f"{what}: mean error {err.mean():.3e} > {mean_bound:.3e}"


def _inputs(M, K, N1, N2, seed, op, b1=True):
    return inputs.b2b_inputs(M, K, N1, N2, seed, x_std=1.0, w1_std=K ** -0.5,
                             w2_std=1.0 if op == "softmax" else N1 ** -0.5, b1_std=0.2 if b1 else None,
                             ln=op == "layernorm")


def _ref(d, op, alpha, rows=None):
    return oracle.b2b_gemm(d["X"], d["W1"], d["W2"], op=op, alpha=alpha, b1=d["b1"], rows=rows,
                           gamma1=d.get("gamma1"), beta1=d.get("beta1"), eps=1e-5)


@pytest.mark.parametrize("op,mode", CASES)
@pytest.mark.parametrize("M,K,N1,N2", [(128, 64, 256, 64), (200, 128, 512, 128), (333, 128, 1024, 64),
                                       (257, 192, 2048, 128), (130, 136, 1024, 128), (150, 320, 512, 64)])
def test_b2b_shapes(op, mode, M, K, N1, N2):
    d = _inputs(M, K, N1, N2, seed=M + K + N1 + N2, op=op)
    alpha = K ** -0.5 if op == "softmax" else 1.0
    o = _run(d, op, alpha, tuning=_tuning(mode, N1))
    ref = _ref(d, op, alpha)
    check_b2b(o, ref, d, op, alpha, f"b2b {op} {mode} {M}x{K}x{N1}x{N2}", mode=mode)


@pytest.mark.parametrize("op,mode", CASES)
@pytest.mark.parametrize("kw", [dict(max_clusters=1), dict(max_clusters=3, stages=2), dict(stages=3),
                                dict(max_clusters=2, disable_pdl=1)])
def test_b2b_persistent_tiles(op, mode, kw):
    """Few clusters (CTAs) for many row blocks: each walks several tiles."""
    M, K, N1, N2 = 1000, 256, 1024, 128
    d = _inputs(M, K, N1, N2, seed=17, op=op, b1=False)
    alpha = 0.25 if op == "softmax" else 1.0
    o = _run(d, op, alpha, tuning=_tuning(mode, N1, **kw))
    ref = _ref(d, op, alpha)
    check_b2b(o, ref, d, op, alpha, f"b2b {op} {mode} {kw}", mode=mode)


@pytest.mark.parametrize("op", ["softmax", "gelu_tanh", "layernorm"])
@pytest.mark.parametrize("M,K,N1,N2,kw", [(300, 128, 4096, 128, {}), (129, 512, 768, 64, {}),
                                          (640, 1024, 512, 128, dict(max_clusters=2)),
                                          (256, 72, 256, 64, dict(stages=3))])
def test_b2b_stream_only_shapes(op, M, K, N1, N2, kw):
    """Stream kernel beyond the cluster kernel's reach (N1 > 8 * 256, N1 not
    a power-of-two multiple of 256) and with X streamed next to W1 (K > 256)."""
    d = _inputs(M, K, N1, N2, seed=M + 3 * K + N1, op=op)
    alpha = K ** -0.5 if op == "softmax" else 1.0
    o = _run(d, op, alpha, tuning=_tuning("stream", N1, **kw))
    ref = _ref(d, op, alpha)
    check_b2b(o, ref, d, op, alpha, f"b2b stream {op} {M}x{K}x{N1}x{N2} {kw}", mode="stream")


@pytest.mark.parametrize("ramp", [0.0, 0.05, -0.05, 1.0])
def test_b2b_stream_softmax_rescaling(ramp):
    """Row maxima that rise (or fall) from chunk to chunk: b1 ramps with the
    column, so later chunks pass the running reference by more than 2^8 and
    the online softmax rescales O and the row sum (ramp 1.0: a rise of about
    128 per chunk in log2 units, every chunk)."""
    M, K, N1, N2 = 256, 128, 2048, 128
    d = _inputs(M, K, N1, N2, seed=31, op="softmax")
    d["b1"] = (d["b1"] + ramp * np.arange(N1)).astype(np.float32)
    alpha = K ** -0.5
    o = _run(d, "softmax", alpha, tuning=_tuning("stream", N1))
    ref = _ref(d, "softmax", alpha)
    check_b2b(o, ref, d, "softmax", alpha, f"b2b stream rescale {ramp}", mode="stream")


@pytest.mark.parametrize("offset,ramp", [(40.0, 0.0), (0.0, 6.0), (-25.0, -3.0)])
def test_b2b_stream_layernorm_shifted_rows(offset, ramp):
    """Rows whose mean is far from 0 (b1 offset) and whose first chunk's mean
    is far from the row's (b1 ramps over N1): the stream kernel's shift mu0
    and its correction -(mu - mu0) rstd gamma1^T W2 are exercised, and the
    normalised result must not lose the precision of the row's spread."""
    M, K, N1, N2 = 384, 128, 1024, 128
    d = _inputs(M, K, N1, N2, seed=71, op="layernorm")
    d["b1"] = (np.asarray(d["b1"], np.float64) + offset + ramp * np.linspace(-1.0, 1.0, N1)).astype(np.float32)
    o = _run(d, "layernorm", 1.0, tuning=_tuning("stream", N1))
    ref = _ref(d, "layernorm", 1.0)
    check_b2b(o, ref, d, "layernorm", 1.0, f"stream LayerNorm offset {offset} ramp {ramp}", mode="stream")


def test_b2b_kernels_agree_on_gelu():
    """GELU rounds the same value in both kernels: outputs within fp32
    accumulation-order noise of each other (the sums over N1 run in a
    different order)."""
    M, K, N1, N2 = 384, 128, 1024, 128
    d = _inputs(M, K, N1, N2, seed=37, op="gelu_tanh")
    a = _run(d, "gelu_tanh", 1.0, tuning=_tuning("cluster", N1))
    b = _run(d, "gelu_tanh", 1.0, tuning=_tuning("stream", N1))
    A, _, _, _ = _terms(d, "gelu_tanh", 1.0)
    bound = 2 * bf16_half_ulp(np.abs(a) + N1 * 2.0 ** -23 * A) + N1 * 2.0 ** -23 * A
    assert np.all(np.abs(a - b) <= bound)


@pytest.mark.parametrize("op,mode", CASES)
@pytest.mark.parametrize("N1,N2", [(256, 64), (2048, 128)])
def test_b2b_selector_reads_back_s(op, mode, N1, N2):
    """W2 with a single 1 per column: O[:, k] = bf16(S[:, c_k]) exactly up to
    the one-ulp rounding difference of S, for columns c_k spread over every
    CTA of the cluster and every position of the packed bf16 pairs."""
    M, K = 256, 128
    d = _inputs(M, K, N1, N2, seed=23, op=op)
    cols = (np.arange(N2) * (N1 // N2) + (np.arange(N2) * 7) % (N1 // N2)) % N1
    W2 = np.zeros((N1, N2), np.float32)
    W2[cols, np.arange(N2)] = 1.0
    d["W2"] = W2
    alpha = K ** -0.5
    o = _run(d, op, alpha, tuning=_tuning(mode, N1))
    z = alpha * oracle.gemm(d["X"], d["W1"]) + np.asarray(d["b1"], np.float64)
    s = _s(d, op, z)
    sel = s[:, cols]
    e = 2.0 ** -16 * np.abs(sel) + (0.5 * 2.0 ** -10.98 * np.abs(z[:, cols]) if op == "gelu_tanh" else 0.0)
    if op == "layernorm":
        e = e + 2.0 ** -14 * (np.abs(sel) + 1.0)
    bound = 2 * bf16_half_ulp(np.abs(sel) + e) + e
    if mode == "stream" and op == "softmax":
        # the unnormalised exponential is rounded (relative error <= 2^-8), then
        # the output: one bf16 rounding more than the cluster kernel's
        bound = bf16_half_ulp(np.abs(sel) + e) + 2.0 ** -8 * (np.abs(sel) + e) + e
    if mode == "stream" and op == "layernorm":
        # (z - mu0) gamma1 is rounded (relative error <= 2^-9 of |t|), then the output
        t = np.abs(_shifted(d, z)[:, cols])
        bound = bf16_half_ulp(np.abs(sel) + 2.0 ** -8 * t + e) + 2.0 ** -8 * t + e
    err = np.abs(o - sel)
    worst = np.argmax(err - bound)
    assert err.flat[worst] <= bound.flat[worst], (
        f"selector {op}: error {err.flat[worst]:.3e} > {bound.flat[worst]:.3e} (col {cols[worst % N2]})")


@pytest.mark.parametrize("op", ["softmax", "layernorm"])
def test_b2b_stream_timeout_is_reported(op):
    """One more arrival at the P-ready barrier than can happen: the MMA warp's
    bounded wait runs out (or the producer's, blocked behind it, first), the
    kernel records CF_ERR_DEVICE_TIMEOUT with the role and every role drains
    (LayerNorm: with its fold kernel before it); the context stays usable."""
    M, K, N1, N2 = 512, 128, 512, 128
    d = _inputs(M, K, N1, N2, seed=43, op=op)
    alpha = K ** -0.5
    torch = torch_cuda()
    X, W1, W2 = dev_bf16(d["X"]), dev_bf16(d["W1"]), dev_bf16(d["W2"])
    b1 = dev_f32(d["b1"])
    O = torch.zeros((M, N2), dtype=torch.bfloat16, device="cuda")
    ws = cf.new_workspace(cf.cf_b2b_workspace_size())
    t = _tuning("stream", N1, extra_arrivals=1, timeout_us=2000)
    if op == "layernorm":
        st = cf.cf_b2b_gemm_layernorm(X, W1, b1, dev_f32(d["gamma1"]), dev_f32(d["beta1"]), W2, O, M, K, N1, N2,
                                      alpha, 1e-5, ws, ws.numel(), None, t)
    else:
        st = cf.cf_b2b_gemm(X, W1, b1, W2, O, M, K, N1, N2, alpha, cf.CF_B2B_SOFTMAX, ws, ws.numel(), None, t)
    assert st == cf.CF_OK
    dst, info = cf.cf_get_device_status(ws)
    assert dst == cf.CF_ERR_DEVICE_TIMEOUT
    info &= 0xFFFFFFFF  # (the binding returns the word signed)
    assert (info >> 24) in (0x91, 0x92, 0x93), hex(info)  # a wait of the stream kernel's roles
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK  # cleared by the read
    o = _run(d, op, alpha, tuning=_tuning("stream", N1))
    check_b2b(o, _ref(d, op, alpha), d, op, alpha, "after a timeout", mode="stream")


def test_b2b_empty_and_unsupported():
    torch = torch_cuda()
    ws = cf.new_workspace(cf.cf_b2b_workspace_size())
    X = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    W1 = torch.zeros((128, 512), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((512, 128), dtype=torch.bfloat16, device="cuda")
    O = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    n = ws.numel()
    assert cf.cf_b2b_gemm(X, W1, None, W2, O, 0, 128, 512, 128, 1.0, 0, ws, n) == cf.CF_OK
    assert cf.cf_b2b_gemm(X, W1, None, W2, O, 128, 128, 384, 128, 1.0, 0, ws, n) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_b2b_gemm(X, W1, None, W2, O, 128, 128, 512, 96, 1.0, 0, ws, n) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_b2b_gemm(X, W1, None, W2, O, 128, 12, 512, 128, 1.0, 0, ws, n) == cf.CF_ERR_UNSUPPORTED
    # N1 = 4096: 16 CTAs per row block is beyond the cluster kernel (the
    # stream kernel has no such limit); a tile width other than 128 (stream)
    # or 256 (cluster)
    g = torch.ones(512, device="cuda")
    assert cf.cf_b2b_gemm_layernorm(X, W1, None, g, g, W2, O, 128, 128, 4096, 128, 1.0, 1e-5, ws, n, None,
                                    cf.tuning(n_slice=256)) == cf.CF_ERR_UNSUPPORTED
    for ns in (64, 192, 512):
        assert cf.cf_b2b_gemm(X, W1, None, W2, O, 128, 128, 512, 128, 1.0, 0, ws, n, None,
                              cf.tuning(n_slice=ns)) == cf.CF_ERR_UNSUPPORTED
    assert cf.cf_b2b_gemm(X, W1, None, W2, O, 128, 128, 512, 128, 1.0, 3, ws, n) == cf.CF_ERR_INVALID_ARG
    # the LayerNorm epilogue needs gamma1 and beta1: only through its own entry point
    assert cf.cf_b2b_gemm(X, W1, None, W2, O, 128, 128, 512, 128, 1.0, 2, ws, n) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm_layernorm(X, W1, None, None, g, W2, O, 128, 128, 512, 128, 1.0, 1e-5, ws,
                                    n) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm(X, W1, None, W2, X, 128, 128, 512, 128, 1.0, 0, ws, n) == cf.CF_ERR_INVALID_ARG
    assert cf.cf_b2b_gemm(X, W1, None, W2, O, 128, 128, 512, 128, 1.0, 0, ws, 16) == cf.CF_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert cf.cf_get_device_status(ws)[0] == cf.CF_OK


def test_b2b_plan():
    torch = torch_cuda()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # the stream kernel is the default: one CTA per SM, 256-column chunks
    st, p = cf.cf_query_b2b_plan(32768, 128, 1024, 128, cf.CF_B2B_SOFTMAX)
    assert st == cf.CF_OK
    assert p.cluster_size == 1 and p.n_slice == 128 and p.row_blocks == 256 and p.clusters == min(256, sms)
    assert 232448 // 2 < p.smem_bytes <= 232448 and p.stages >= 3
    st, p = cf.cf_query_b2b_plan(32768, 128, 1024, 128, cf.CF_B2B_SOFTMAX, cf.tuning(n_slice=256))
    assert st == cf.CF_OK
    assert p.cluster_size == 4 and p.n_slice == 256 and p.row_blocks == 256 and 1 <= p.clusters <= 256
    assert p.clusters * p.cluster_size <= sms and p.smem_bytes <= 232448 and p.stages >= 2
    st, p = cf.cf_query_b2b_plan(100, 64, 2048, 64, cf.CF_B2B_GELU_TANH, cf.tuning(max_clusters=1))
    assert st == cf.CF_OK and p.cluster_size == 1 and p.clusters == 1
    st, p = cf.cf_query_b2b_plan(100, 64, 2048, 64, cf.CF_B2B_LAYERNORM, cf.tuning(n_slice=256))
    assert st == cf.CF_OK and p.cluster_size == 8
    # LayerNorm defaults to the stream kernel too, at any N1
    for N1 in (2048, 4096):
        st, p = cf.cf_query_b2b_plan(100, 64, N1, 64, cf.CF_B2B_LAYERNORM)
        assert st == cf.CF_OK and p.cluster_size == 1 and p.n_slice == 128


@pytest.mark.parametrize("name,mode", [("b2b_attn_32768x128x1024x128", "stream"),
                                       ("b2b_attn_32768x128x1024x128", "cluster"),
                                       ("b2b_gelu_16384x1024x2048x128", "stream"),
                                       ("b2b_gelu_16384x1024x2048x128", "cluster"),
                                       ("b2b_ln_16384x1024x2048x128", "cluster"),
                                       ("b2b_ln_16384x1024x2048x128", "stream")])
def test_b2b_full_workload(name, mode):
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(name)
    o = _run(d, w.op, w.alpha, tuning=_tuning(mode, w.N1))
    rows = sample_rows(w.M, 384, seed=11)
    ref = _ref(d, w.op, w.alpha, rows=rows)
    sub = dict(d, X=d["X"][rows])
    check_b2b(o[rows], ref, sub, w.op, w.alpha, f"{name} {mode}", mode=mode)
