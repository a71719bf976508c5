"""Helpers for the GPU parity tests: device upload of the seeded inputs and the
tolerance checks (max-abs / mean-abs for LayerNorm outputs, max-abs and row-sum
error for softmax outputs), always against the unrounded fp64 oracle."""
import numpy as np
import pytest

LN_MAX_ABS = 2e-2
LN_MEAN_ABS = 2e-3
SM_MAX_ABS = 1e-3
SM_ROWSUM = 1e-2


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def dev_bf16(a):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(torch.bfloat16)


def dev_f32(a):
    torch = torch_cuda()
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def bf16_half_ulp(v):
    """Half a bf16 ulp at |v| (8 mantissa bits incl. the implicit one)."""
    a = np.maximum(np.abs(v), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 8)


def check_ln(y, ref, what="", strict=False):
    """max-abs 2e-2 and mean-abs 2e-3 against the unrounded fp64 oracle.

    Where |ref| >= 8 the bf16 output's own rounding (half an ulp = 1/32) is
    larger than 2e-2, so there the bound is half an ulp plus the 4e-3 the
    2e-2 budget leaves for fp32 arithmetic below |ref| = 8 (2e-2 - 1/64).
    ``strict=True`` asserts that no element needs that allowance.
    """
    err = np.abs(y - ref)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    if strict:
        assert np.abs(ref).max() < 8.0, f"{what}: |ref| reaches {np.abs(ref).max():.3f}"
    bound = np.maximum(LN_MAX_ABS, bf16_half_ulp(ref) + (LN_MAX_ABS - 2.0 ** -6))
    worst = np.argmax(err - bound)
    assert err.flat[worst] <= bound.flat[worst], (
        f"{what}: error {err.flat[worst]:.3e} at |ref|={abs(ref.flat[worst]):.3f} > {bound.flat[worst]:.3e}")
    assert err.mean() <= LN_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e} > {LN_MEAN_ABS}"
    return float(err.max()), float(err.mean())


def check_softmax(y, ref, what="", bf16_out=False, strict=False):
    """max-abs 1e-3 and every row sum within 1e-2 of 1, against the unrounded
    fp64 oracle.

    A bf16 output (``bf16_out``) carries its own rounding: half an ulp exceeds
    1e-3 where |ref| >= 1/2, so there the bound is half an ulp plus the
    2.3e-5 the 1e-3 budget leaves for fp32 arithmetic below 1/2
    (1e-3 - 2^-10).  ``strict=True`` asserts that no element needs it (the
    page workload's outputs are about 1/2048).
    """
    err = np.abs(y - ref)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    if strict:
        assert np.abs(ref).max() < 0.5, f"{what}: |ref| reaches {np.abs(ref).max():.3f}"
    bound = np.maximum(SM_MAX_ABS, bf16_half_ulp(ref) + (SM_MAX_ABS - 2.0 ** -10)) if bf16_out else SM_MAX_ABS
    worst = np.argmax(err - bound)
    bw = bound.flat[worst] if bf16_out else bound
    assert err.flat[worst] <= bw, f"{what}: error {err.flat[worst]:.3e} at |ref|={abs(ref.flat[worst]):.3f} > {bw:.3e}"
    rs = np.abs(y.sum(axis=1) - 1.0)
    assert rs.max() <= SM_ROWSUM, f"{what}: row-sum error {rs.max():.3e} > {SM_ROWSUM}"
    return float(err.max()), float(rs.max())


def sample_rows(M, n, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    rows.update([0, M - 1])
    return np.array(sorted(rows), dtype=np.int64)


def check_ln_all_rows(Y, ref_rows, what="", strict=False, chunk=2048):
    """check_ln over every row of the device output Y [M, N], in row chunks
    (the oracle is row-independent, so each chunk's reference is exact):
    the max-abs bound per element, the mean-abs bound over all M*N elements.
    ``ref_rows(rows)`` returns the oracle's rows ``rows``."""
    M = Y.shape[0]
    tot, n = 0.0, 0
    worst = 0.0
    for r0 in range(0, M, chunk):
        rows = np.arange(r0, min(M, r0 + chunk), dtype=np.int64)
        y = host(Y[r0:r0 + len(rows)])
        ref = ref_rows(rows)
        err = np.abs(y - ref)
        assert np.all(np.isfinite(y)), f"{what}: non-finite output in rows {r0}.."
        if strict:
            assert np.abs(ref).max() < 8.0, f"{what}: |ref| reaches {np.abs(ref).max():.3f}"
        bound = np.maximum(LN_MAX_ABS, bf16_half_ulp(ref) + (LN_MAX_ABS - 2.0 ** -6))
        w = np.argmax(err - bound)
        assert err.flat[w] <= bound.flat[w], (
            f"{what}: error {err.flat[w]:.3e} at row {r0 + w // y.shape[1]} (|ref|={abs(ref.flat[w]):.3f})"
            f" > {bound.flat[w]:.3e}")
        worst = max(worst, float(err.max()))
        tot += float(err.sum())
        n += err.size
    assert n == Y.shape[0] * Y.shape[1]
    assert tot / n <= LN_MEAN_ABS, f"{what}: mean-abs {tot / n:.3e} > {LN_MEAN_ABS}"
    return worst, tot / n
