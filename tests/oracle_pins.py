"""Pin checks for the fp64 oracle, written against what the mathematics fixes.

Each ``check_*`` takes the function under test as an argument and returns a
list of failure strings (empty = pinned).  ``test_oracle_pins.py`` runs them
on the oracle; ``test_oracle_mutations.py`` runs them on deliberately broken
copies (a dropped term, a wrong sign, a transposed operand ...) to show each
plausible mistake fails at least one pin.  Nothing here calls the oracle's
own helpers to compute an expected value: expected values are closed forms,
brute force, hand-derived fixtures or independent library routines.
"""
from __future__ import annotations

import math
import os
import statistics
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([float(v) for v in line.split()])
    return np.array(rows, dtype=np.float64)


def _fail(fails, ok, msg):
    if not ok:
        fails.append(msg)


# ----------------------------------------------------------------------------
# MatMul
# ----------------------------------------------------------------------------
def check_gemm(gemm) -> list:
    fails = []
    rng = np.random.Generator(np.random.PCG64(11))
    # brute force with exact rational arithmetic on small integer matrices
    for (M, K, N) in [(3, 5, 7), (4, 2, 9), (1, 6, 1), (5, 1, 3)]:
        X = rng.integers(-8, 9, size=(M, K))
        W = rng.integers(-8, 9, size=(K, N))
        exact = np.array([[sum(Fraction(int(X[i, k])) * int(W[k, j]) for k in range(K))
                           for j in range(N)] for i in range(M)], dtype=np.float64)
        P = np.asarray(gemm(X.astype(np.float64), W.astype(np.float64)))
        _fail(fails, P.shape == (M, N), f"gemm shape {P.shape} != {(M, N)}")
        _fail(fails, P.shape == (M, N) and np.array_equal(P, exact),
              f"gemm {M}x{K}x{N} integer product not exact")
    # bf16-valued reals: products exact in fp64; compare with a Python loop
    X = np.round(rng.standard_normal((6, 10)) * 64) / 64
    W = np.round(rng.standard_normal((10, 4)) * 64) / 64
    ref = np.array([[math.fsum(X[i, k] * W[k, j] for k in range(10)) for j in range(4)]
                    for i in range(6)])
    P = np.asarray(gemm(X, W))
    _fail(fails, P.shape == ref.shape and np.allclose(P, ref, rtol=1e-13, atol=1e-13),
          "gemm real-valued mismatch vs fsum brute force")
    return fails


# ----------------------------------------------------------------------------
# GELU (tanh form)
# ----------------------------------------------------------------------------
def check_gelu(gelu) -> list:
    fails = []
    _fail(fails, float(np.asarray(gelu(np.array([0.0])))[0]) == 0.0, "GELU(0) != 0")
    x = np.linspace(-6, 6, 241)
    g = np.asarray(gelu(x))
    gm = np.asarray(gelu(-x))
    # tanh is odd: GELU(x) - GELU(-x) = x exactly up to rounding
    _fail(fails, np.allclose(g - gm, x, rtol=1e-14, atol=1e-14), "GELU(x)-GELU(-x) != x")
    # asymptotes
    _fail(fails, abs(float(np.asarray(gelu(np.array([12.0])))[0]) - 12.0) < 1e-12, "GELU(12) != 12")
    _fail(fails, abs(float(np.asarray(gelu(np.array([-12.0])))[0])) < 1e-12, "GELU(-12) != 0")
    # second-order coefficient: (GELU(h)+GELU(-h))/(2h^2) -> sqrt(2/pi)/2
    h = 1e-4
    even = (float(np.asarray(gelu(np.array([h])))[0]) + float(np.asarray(gelu(np.array([-h])))[0])) / (2 * h * h)
    _fail(fails, abs(even - math.sqrt(2 / math.pi) / 2) < 1e-6, f"GELU curvature {even}")
    # independent library routine (fp64)
    import torch
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    _fail(fails, np.allclose(g, ref, rtol=1e-13, atol=1e-15), "GELU vs torch gelu(tanh) fp64")
    return fails


# ----------------------------------------------------------------------------
# LayerNorm
# ----------------------------------------------------------------------------
def check_layernorm(ln) -> list:
    fails = []
    rng = np.random.Generator(np.random.PCG64(12))
    # eps = 0, gamma = 1, beta = 0: row mean 0 and (biased) variance 1 to 1e-9
    for N in (2, 3, 7, 512, 4096):
        g = rng.standard_normal((5, N)) * 0.013 + 0.37
        y = np.asarray(ln(g, np.ones(N), np.zeros(N), 0.0))
        mean = y.mean(axis=1)
        var = ((y - y.mean(axis=1, keepdims=True)) ** 2).mean(axis=1)
        _fail(fails, np.all(np.abs(mean) < 1e-9), f"LN eps=0 mean N={N}: {mean}")
        _fail(fails, np.all(np.abs(var - 1) < 1e-9), f"LN eps=0 var N={N}: {var}")
    # eps > 0: output variance = s2/(s2+eps), s2 from Python's statistics module
    for N in (4, 33):
        row = rng.standard_normal(N) * 0.01
        s2 = statistics.pvariance([float(v) for v in row])
        eps = 1e-5
        y = np.asarray(ln(row[None, :], np.ones(N), np.zeros(N), eps))[0]
        v = float(((y - y.mean()) ** 2).mean())
        _fail(fails, abs(v - s2 / (s2 + eps)) < 1e-9, f"LN eps>0 var {v} vs {s2 / (s2 + eps)}")
    # constant row -> beta exactly
    N = 16
    beta = rng.standard_normal(N)
    y = np.asarray(ln(np.full((1, N), 3.25), rng.standard_normal(N), beta, 1e-5))[0]
    _fail(fails, np.array_equal(y, beta), "LN constant row != beta")
    # two elements [a, b]: y = [-d, d]/sqrt(d^2+eps) with d = (b-a)/2
    a, b, eps = 0.3, -1.1, 1e-3
    d = (b - a) / 2
    y = np.asarray(ln(np.array([[a, b]]), np.ones(2), np.zeros(2), eps))[0]
    want = np.array([-d, d]) / math.sqrt(d * d + eps)
    _fail(fails, np.allclose(y, want, rtol=1e-13, atol=1e-15), "LN two-element closed form")
    # positive row scaling leaves the result unchanged at eps = 0
    g = rng.standard_normal((3, 64))
    y1 = np.asarray(ln(g, np.ones(64), np.zeros(64), 0.0))
    y2 = np.asarray(ln(g * 37.5, np.ones(64), np.zeros(64), 0.0))
    _fail(fails, np.allclose(y1, y2, rtol=1e-12, atol=1e-12), "LN scale invariance")
    # hand-derived worked fixture (gamma/beta affine after normalising)
    t = _load_golden("layernorm_worked.txt")
    for blk in (t[:4], t[4:]):
        g, gam, bet, eps, want = blk[:, 0], blk[:, 1], blk[:, 2], blk[0, 3], blk[:, 4]
        y = np.asarray(ln(g[None, :], gam, bet, eps))[0]
        _fail(fails, np.allclose(y, want, rtol=1e-12, atol=1e-12), f"LN golden {y} vs {want}")
    # independent library routine (fp64)
    import torch
    g = rng.standard_normal((4, 96)) * 0.02
    gam = 1 + 0.1 * rng.standard_normal(96)
    bet = 0.1 * rng.standard_normal(96)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(g), (96,), torch.from_numpy(gam),
                                         torch.from_numpy(bet), 1e-5).numpy()
    y = np.asarray(ln(g, gam, bet, 1e-5))
    _fail(fails, np.allclose(y, ref, rtol=1e-11, atol=1e-12), "LN vs torch layer_norm fp64")
    return fails


# ----------------------------------------------------------------------------
# RMSNorm
# ----------------------------------------------------------------------------
def check_rmsnorm(rms) -> list:
    fails = []
    rng = np.random.Generator(np.random.PCG64(16))
    # eps = 0, gamma = 1, no beta: every row's mean square is 1 to 1e-12
    for N in (1, 2, 7, 512, 4096):
        g = rng.standard_normal((5, N)) * 0.013 + 0.37
        y = np.asarray(rms(g, np.ones(N), None, 0.0))
        ms = (y * y).mean(axis=1)
        _fail(fails, np.all(np.abs(ms - 1) < 1e-12), f"RMS eps=0 mean square N={N}: {ms}")
    # the mean is not subtracted: a row with a large offset keeps its sign pattern
    g = np.array([[10.0, 10.5, 9.5]])
    y = np.asarray(rms(g, np.ones(3), None, 0.0))[0]
    _fail(fails, np.all(y > 0), "RMS keeps the mean (no centring)")
    # eps > 0: output mean square = ms / (ms + eps), ms by exact summation of squares
    for N in (4, 33):
        row = rng.standard_normal(N) * 0.01
        ms = math.fsum(float(v) * float(v) for v in row) / N
        eps = 1e-5
        y = np.asarray(rms(row[None, :], np.ones(N), None, eps))[0]
        _fail(fails, abs(float((y * y).mean()) - ms / (ms + eps)) < 1e-12, "RMS eps>0 mean square")
    # constant row c: y = c / sqrt(c^2 + eps) * gamma + beta
    N, c, eps = 8, -2.5, 0.25
    gam = rng.standard_normal(N)
    bet = rng.standard_normal(N)
    y = np.asarray(rms(np.full((1, N), c), gam, bet, eps))[0]
    _fail(fails, np.allclose(y, c / math.sqrt(c * c + eps) * gam + bet, rtol=1e-14, atol=1e-15), "RMS constant row")
    # odd under sign flip, invariant under positive scaling at eps = 0
    g = rng.standard_normal((3, 64))
    y1 = np.asarray(rms(g, np.ones(64), None, 0.0))
    _fail(fails, np.allclose(np.asarray(rms(-g, np.ones(64), None, 0.0)), -y1, rtol=0, atol=1e-15), "RMS sign")
    _fail(fails, np.allclose(np.asarray(rms(g * 37.5, np.ones(64), None, 0.0)), y1, rtol=1e-12, atol=1e-12),
          "RMS scale invariance")
    # beta None == beta 0
    _fail(fails, np.array_equal(np.asarray(rms(g, np.ones(64), None, 1e-5)),
                                np.asarray(rms(g, np.ones(64), np.zeros(64), 1e-5))), "RMS beta None")
    # hand-derived worked fixture
    t = _load_golden("rmsnorm_worked.txt")
    for blk in (t[:2], t[2:]):
        g, gam, bet, eps, want = blk[:, 0], blk[:, 1], blk[:, 2], blk[0, 3], blk[:, 4]
        y = np.asarray(rms(g[None, :], gam, bet, eps))[0]
        _fail(fails, np.allclose(y, want, rtol=1e-13, atol=1e-15), f"RMS golden {y} vs {want}")
    # independent library routine (fp64)
    import torch
    g = rng.standard_normal((4, 96)) * 0.02
    gam = 1 + 0.1 * rng.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(g), (96,), torch.from_numpy(gam), 1e-5).numpy()
    _fail(fails, np.allclose(np.asarray(rms(g, gam, None, 1e-5)), ref, rtol=1e-11, atol=1e-12),
          "RMS vs torch rms_norm fp64")
    return fails


def check_rmsnorm_composition(fused) -> list:
    import torch
    F = torch.nn.functional
    fails = []
    rng = np.random.Generator(np.random.PCG64(17))
    M, K, N = 9, 24, 40
    X = rng.standard_normal((M, K)) / 5
    W = rng.standard_normal((K, N)) / 5
    bias = rng.standard_normal(N) * 0.1
    gam = 1 + rng.standard_normal(N) * 0.1
    bet = rng.standard_normal(N) * 0.1
    t = {k: torch.from_numpy(v) for k, v in dict(X=X, W=W, b=bias, g=gam, be=bet).items()}
    for act in ("none", "gelu_tanh"):
        for alpha in (1.0, 0.5):
            x = alpha * (t["X"] @ t["W"]) + t["b"]
            if act == "gelu_tanh":
                x = F.gelu(x, approximate="tanh")
            ref = (F.rms_norm(x, (N,), t["g"], 1e-5) + t["be"]).numpy()
            y = np.asarray(fused(X, W, bias, gam, bet, alpha=alpha, eps=1e-5, act=act))
            _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-10, atol=1e-11),
                  f"rmsnorm composition act={act} alpha={alpha}")
    y0 = np.asarray(fused(X, W, None, gam, None, alpha=1.0, eps=1e-5, act="none"))
    y1 = np.asarray(fused(X, W, np.zeros(N), gam, np.zeros(N), alpha=1.0, eps=1e-5, act="none"))
    _fail(fails, np.allclose(y0, y1, rtol=0, atol=1e-15), "rmsnorm bias/beta None")
    rows = [8, 0, 3]
    ys = np.asarray(fused(X, W, bias, gam, bet, alpha=1.0, eps=1e-5, act="gelu_tanh", rows=rows))
    yf = np.asarray(fused(X, W, bias, gam, bet, alpha=1.0, eps=1e-5, act="gelu_tanh"))
    _fail(fails, ys.shape == yf[rows].shape and np.allclose(ys, yf[rows], rtol=1e-13, atol=1e-14),
          "rmsnorm rows= subset")
    return fails


def check_residual_norm(fused) -> list:
    """Residual add + norm: torch compositions in fp64; R = 0 is the plain call;
    LayerNorm is invariant to a constant added to every column of a row, so a
    per-row constant residual changes nothing; the residual enters after GELU."""
    import torch
    F = torch.nn.functional
    import oracle
    fails = []
    rng = np.random.Generator(np.random.PCG64(18))
    M, K, N = 9, 24, 40
    X = rng.standard_normal((M, K)) / 5
    W = rng.standard_normal((K, N)) / 5
    R = rng.standard_normal((M, N)) * 0.3
    bias = rng.standard_normal(N) * 0.1
    gam = 1 + rng.standard_normal(N) * 0.1
    bet = rng.standard_normal(N) * 0.1
    t = {k: torch.from_numpy(v) for k, v in dict(X=X, W=W, R=R, b=bias, g=gam, be=bet).items()}
    for act in ("none", "gelu_tanh"):
        for norm in ("layer", "rms"):
            x = 0.5 * (t["X"] @ t["W"]) + t["b"]
            if act == "gelu_tanh":
                x = F.gelu(x, approximate="tanh")
            g = x + t["R"]
            ref = (F.layer_norm(g, (N,), t["g"], t["be"], 1e-5) if norm == "layer"
                   else F.rms_norm(g, (N,), t["g"], 1e-5) + t["be"]).numpy()
            y = np.asarray(fused(X, W, bias, R, gam, bet, alpha=0.5, eps=1e-5, act=act, norm=norm))
            _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-10, atol=1e-11),
                  f"residual composition act={act} norm={norm}")
    y0 = np.asarray(fused(X, W, bias, np.zeros((M, N)), gam, bet, eps=1e-5, act="gelu_tanh", norm="layer"))
    y1 = oracle.gemm_bias_rownorm(X, W, bias, gam, bet, eps=1e-5, act="gelu_tanh")
    _fail(fails, np.allclose(y0, y1, rtol=1e-13, atol=1e-14), "residual R=0 is the plain LayerNorm call")
    shift = np.repeat(rng.standard_normal((M, 1)) * 5, N, axis=1)
    y2 = np.asarray(fused(X, W, bias, shift, gam, bet, eps=0.0, act="none", norm="layer"))
    y3 = np.asarray(fused(X, W, bias, np.zeros((M, N)), gam, bet, eps=0.0, act="none", norm="layer"))
    _fail(fails, np.allclose(y2, y3, rtol=1e-9, atol=1e-10), "LayerNorm ignores a per-row constant residual")
    rows = [8, 0, 3]
    ys = np.asarray(fused(X, W, bias, R, gam, None, act="none", norm="rms", rows=rows))
    yf = np.asarray(fused(X, W, bias, R, gam, None, act="none", norm="rms"))
    _fail(fails, np.allclose(ys, yf[rows], rtol=1e-13, atol=1e-14), "residual rows= subset")
    return fails


# ----------------------------------------------------------------------------
# Softmax
# ----------------------------------------------------------------------------
def check_softmax(sm) -> list:
    fails = []
    rng = np.random.Generator(np.random.PCG64(13))
    z = rng.standard_normal((6, 2048)) * 3
    y = np.asarray(sm(z))
    _fail(fails, np.all(np.abs(y.sum(axis=1) - 1) < 1e-12), "softmax rows do not sum to 1")
    _fail(fails, np.all(y > 0), "softmax not positive")
    # invariance to a per-row constant shift
    shift = rng.standard_normal((6, 1)) * 50
    y2 = np.asarray(sm(z + shift))
    _fail(fails, np.allclose(y, y2, rtol=1e-11, atol=1e-16), "softmax shift invariance")
    # large magnitudes must not overflow (the max subtraction is part of it)
    big = np.array([[1000.0, 999.0, 998.0]])
    yb = np.asarray(sm(big))
    _fail(fails, bool(np.all(np.isfinite(yb))) and abs(float(yb.sum()) - 1) < 1e-12,
          "softmax overflow at large logits")
    # constant row -> 1/N; N = 1 -> 1
    _fail(fails, np.allclose(np.asarray(sm(np.full((1, 37), -4.5))), 1 / 37, rtol=1e-14), "softmax const row")
    _fail(fails, float(np.asarray(sm(np.array([[7.0]])))[0, 0]) == 1.0, "softmax N=1")
    # two elements: sigmoid closed form, base e
    a, b = 0.25, 1.75
    y = np.asarray(sm(np.array([[a, b]])))[0]
    _fail(fails, abs(y[0] - 1 / (1 + math.exp(b - a))) < 1e-15, "softmax two-element closed form")
    # argmax preserved
    _fail(fails, np.array_equal(np.argmax(np.asarray(sm(z)), 1), np.argmax(z, 1)), "softmax argmax")
    # hand-derived fixture
    t = _load_golden("softmax_worked.txt")
    for off in (0.0, 100.0):
        y = np.asarray(sm(t[None, :, 0] + off))[0]
        _fail(fails, np.allclose(y, t[:, 1], rtol=1e-13), f"softmax golden (offset {off})")
    import torch
    ref = torch.softmax(torch.from_numpy(z), dim=1).numpy()
    _fail(fails, np.allclose(np.asarray(sm(z)), ref, rtol=1e-12, atol=1e-18), "softmax vs torch fp64")
    return fails


# ----------------------------------------------------------------------------
# Compositions (library cross-check of the wiring: alpha, bias, act, norm)
# ----------------------------------------------------------------------------
def check_rownorm_composition(fused) -> list:
    import torch
    F = torch.nn.functional
    fails = []
    rng = np.random.Generator(np.random.PCG64(14))
    M, K, N = 9, 24, 40
    X = rng.standard_normal((M, K)) / 5
    W = rng.standard_normal((K, N)) / 5
    bias = rng.standard_normal(N) * 0.1
    gam = 1 + rng.standard_normal(N) * 0.1
    bet = rng.standard_normal(N) * 0.1
    t = {k: torch.from_numpy(v) for k, v in dict(X=X, W=W, b=bias, g=gam, be=bet).items()}
    for act in ("none", "gelu_tanh"):
        for alpha in (1.0, 0.5):
            x = alpha * (t["X"] @ t["W"]) + t["b"]
            if act == "gelu_tanh":
                x = F.gelu(x, approximate="tanh")
            ref = F.layer_norm(x, (N,), t["g"], t["be"], 1e-5).numpy()
            y = np.asarray(fused(X, W, bias, gam, bet, alpha=alpha, eps=1e-5, act=act))
            _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-10, atol=1e-11),
                  f"rownorm composition act={act} alpha={alpha}")
    # bias=None is the same as a zero bias
    y0 = np.asarray(fused(X, W, None, gam, bet, alpha=1.0, eps=1e-5, act="none"))
    y1 = np.asarray(fused(X, W, np.zeros(N), gam, bet, alpha=1.0, eps=1e-5, act="none"))
    _fail(fails, np.allclose(y0, y1, rtol=0, atol=1e-15), "rownorm bias=None")
    # sampled rows == the same rows of the full result
    rows = [8, 0, 3]
    ys = np.asarray(fused(X, W, bias, gam, bet, alpha=1.0, eps=1e-5, act="gelu_tanh", rows=rows))
    yf = np.asarray(fused(X, W, bias, gam, bet, alpha=1.0, eps=1e-5, act="gelu_tanh"))
    _fail(fails, ys.shape == yf[rows].shape and np.allclose(ys, yf[rows], rtol=1e-13, atol=1e-14), "rownorm rows= subset")
    return fails


def check_softmax_composition(fused) -> list:
    import torch
    fails = []
    rng = np.random.Generator(np.random.PCG64(15))
    M, K, N = 7, 16, 33
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N)) / 4
    bias = rng.standard_normal(N)
    for b in (None, bias):
        z = 0.3 * (torch.from_numpy(X) @ torch.from_numpy(W))
        if b is not None:
            z = z + torch.from_numpy(b)
        ref = torch.softmax(z, dim=1).numpy()
        y = np.asarray(fused(X, W, scale=0.3, bias=b))
        _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-12, atol=1e-16),
              f"softmax composition bias={'yes' if b is not None else 'no'}")
    rows = [6, 2]
    ys = np.asarray(fused(X, W, scale=0.3, rows=rows))
    yf = np.asarray(fused(X, W, scale=0.3))[rows]
    _fail(fails, ys.shape == yf.shape and np.allclose(ys, yf, rtol=1e-13, atol=1e-18), "softmax rows= subset")
    return fails


def check_softmax_causal(fused) -> list:
    """Causal softmax: torch's softmax over masked_fill(-inf) in fp64; an offset at
    least N - 1 is the unmasked call; masked entries are exactly 0 and kept rows
    sum to 1; a fully masked row is 0; a row keeping one element puts 1 there."""
    import torch
    import oracle
    fails = []
    rng = np.random.Generator(np.random.PCG64(19))
    M, K, N = 12, 16, 20
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N)) / 4
    bias = rng.standard_normal(N)
    for off in (0, 3, -2):
        for b in (None, bias):
            z = 0.7 * (torch.from_numpy(X) @ torch.from_numpy(W))
            if b is not None:
                z = z + torch.from_numpy(b)
            keep = torch.arange(N)[None, :] <= (torch.arange(M)[:, None] + off)
            ref = torch.softmax(z.masked_fill(~keep, float("-inf")), dim=1)
            ref = torch.nan_to_num(ref, nan=0.0).numpy()
            y = np.asarray(fused(X, W, scale=0.7, offset=off, bias=b))
            _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-12, atol=1e-16),
                  f"causal softmax offset={off} bias={'yes' if b is not None else 'no'}")
            k = keep.numpy()
            _fail(fails, np.all(y[~k] == 0.0), f"causal masked entries are 0 (offset {off})")
            live = k.any(axis=1)
            _fail(fails, np.allclose(y[live].sum(1), 1.0, rtol=0, atol=1e-12), f"causal kept rows sum to 1 ({off})")
            _fail(fails, np.all(y[~live] == 0.0), f"causal fully masked rows are 0 ({off})")
    y = np.asarray(fused(X, W, scale=0.7, offset=N - 1))
    _fail(fails, np.allclose(y, oracle.gemm_rowsoftmax(X, W, scale=0.7), rtol=1e-13, atol=1e-16),
          "causal offset N-1 is the unmasked softmax")
    y = np.asarray(fused(X, W, scale=0.7, offset=-5))
    _fail(fails, y[5, 0] == 1.0 and np.all(y[5, 1:] == 0.0) and np.all(y[:5] == 0.0), "causal one kept element")
    rows = [11, 0, 4]
    ys = np.asarray(fused(X, W, scale=0.7, offset=1, rows=rows))
    yf = np.asarray(fused(X, W, scale=0.7, offset=1))[rows]
    _fail(fails, np.allclose(ys, yf, rtol=1e-13, atol=1e-18), "causal rows= subset")
    return fails


def check_b2b(fused) -> list:
    """B2BGEMM: torch fp64 compositions with the intermediate cast to bf16 by
    torch (softmax, GELU, LayerNorm); W2 = identity returns bf16(S); the
    LayerNorm rows are normalised; linearity in W2."""
    import torch
    F = torch.nn.functional
    fails = []
    rng = np.random.Generator(np.random.PCG64(20))
    M, K, N1, N2 = 7, 16, 24, 10
    X = rng.standard_normal((M, K))
    W1 = rng.standard_normal((K, N1)) / 4
    W2 = rng.standard_normal((N1, N2))
    b1 = rng.standard_normal(N1) * 0.1
    t = {k: torch.from_numpy(v) for k, v in dict(X=X, W1=W1, W2=W2, b=b1).items()}
    for op in ("softmax", "gelu_tanh"):
        z = 0.5 * (t["X"] @ t["W1"]) + t["b"]
        S = torch.softmax(z, dim=1) if op == "softmax" else F.gelu(z, approximate="tanh")
        S = S.to(torch.float32).to(torch.bfloat16).to(torch.float64)
        ref = (S @ t["W2"]).numpy()
        y = np.asarray(fused(X, W1, W2, op=op, alpha=0.5, b1=b1))
        _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-12, atol=1e-13), f"b2b {op} vs torch")
        # identity W2 returns the rounded intermediate itself
        I = np.eye(N1)
        yi = np.asarray(fused(X, W1, I, op=op, alpha=0.5, b1=b1))
        _fail(fails, np.array_equal(yi, S.numpy()), f"b2b {op} identity W2")
    # F = LayerNorm over N1 with per-column gamma1, beta1
    g1 = 1 + 0.3 * rng.standard_normal(N1)
    be1 = 0.2 * rng.standard_normal(N1)
    z = 0.5 * (t["X"] @ t["W1"]) + t["b"]
    S = F.layer_norm(z, (N1,), torch.from_numpy(g1), torch.from_numpy(be1), 1e-5)
    S = S.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    ref = (S @ t["W2"]).numpy()
    y = np.asarray(fused(X, W1, W2, op="layernorm", alpha=0.5, b1=b1, gamma1=g1, beta1=be1, eps=1e-5))
    _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-12, atol=1e-13), "b2b layernorm vs torch")
    yi = np.asarray(fused(X, W1, np.eye(N1), op="layernorm", alpha=0.5, b1=b1, gamma1=g1, beta1=be1, eps=1e-5))
    _fail(fails, np.array_equal(yi, S.numpy()), "b2b layernorm identity W2")
    # at eps = 0, gamma = 1, beta = 0 the rounded S rows have mean ~0 and variance ~1
    y1 = np.asarray(fused(X, W1, np.eye(N1), op="layernorm", gamma1=np.ones(N1), beta1=np.zeros(N1), eps=0.0))
    _fail(fails, np.all(np.abs(y1.mean(axis=1)) < 1e-2) and
          all(abs(statistics.pvariance(r) - 1) < 1e-2 for r in y1.tolist()), "b2b layernorm normalised rows")
    # linearity in W2
    W2b = rng.standard_normal((N1, N2))
    y1 = np.asarray(fused(X, W1, W2 + 2.0 * W2b, op="softmax"))
    y2 = np.asarray(fused(X, W1, W2, op="softmax")) + 2.0 * np.asarray(fused(X, W1, W2b, op="softmax"))
    _fail(fails, np.allclose(y1, y2, rtol=1e-12, atol=1e-12), "b2b linear in W2")
    rows = [6, 1]
    ys = np.asarray(fused(X, W1, W2, op="gelu_tanh", rows=rows))
    yf = np.asarray(fused(X, W1, W2, op="gelu_tanh"))[rows]
    _fail(fails, np.allclose(ys, yf, rtol=1e-13, atol=1e-14), "b2b rows= subset")
    return fails


def check_stitch_add_layernorm(fn) -> list:
    """out = LN(A + R) * gamma + beta per row: torch layer_norm in fp64, R
    optional, a hand-derived row, mean 0 / variance 1 at eps = 0, A and R
    interchangeable, a per-row constant in R changes nothing, rows= sampling."""
    import torch
    fails = []
    rng = np.random.Generator(np.random.PCG64(31))
    M, N = 9, 37
    A = rng.standard_normal((M, N)) * 2
    R = rng.standard_normal((M, N))
    g = 1 + 0.3 * rng.standard_normal(N)
    b = 0.2 * rng.standard_normal(N)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(A + R), (N,), torch.from_numpy(g), torch.from_numpy(b),
                                         1e-5).numpy()
    y = np.asarray(fn(A, R, g, b, 1e-5))
    _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-12, atol=1e-12), "add+LN vs torch layer_norm")
    y0 = np.asarray(fn(A, None, g, b, 1e-5))
    yz = np.asarray(fn(A, np.zeros_like(A), g, b, 1e-5))
    _fail(fails, np.array_equal(y0, yz), "add+LN: R = None equals R = 0")
    # hand-derived: x = [2, 2, 4, 4] -> mean 3, variance 1 -> [-1, -1, 1, 1] * gamma + beta
    yh = np.asarray(fn(np.array([[1.0, 2, 3, 4]]), np.array([[1.0, 0, 1, 0]]), np.array([1.0, 2, 3, 4]),
                       np.array([0.0, 0, 0, 1]), 0.0))[0]
    _fail(fails, np.allclose(yh, [-1, -2, 3, 5], rtol=0, atol=1e-15), "add+LN hand-derived row")
    yn = np.asarray(fn(A, R, np.ones(N), np.zeros(N), 0.0))
    _fail(fails, np.all(np.abs(yn.mean(axis=1)) < 1e-12), "add+LN rows have mean 0 at eps = 0")
    _fail(fails, all(abs(statistics.pvariance(r) - 1) < 1e-9 for r in yn.tolist()), "add+LN rows have variance 1")
    _fail(fails, np.allclose(np.asarray(fn(R, A, g, b, 1e-5)), y, rtol=1e-13, atol=1e-13), "add+LN: A + R = R + A")
    shift = rng.standard_normal((M, 1)) * 5
    _fail(fails, np.allclose(np.asarray(fn(A, R + shift, g, b, 1e-5)), y, rtol=1e-9, atol=1e-9),
          "add+LN invariant under a per-row constant in R")
    rows = [7, 0, 3]
    _fail(fails, np.allclose(np.asarray(fn(A, R, g, b, 1e-5, rows=rows)), y[rows], rtol=1e-14, atol=1e-14),
          "add+LN rows= subset")
    return fails


def check_stitch_batchnorm(fn) -> list:
    """BatchNorm over rows: torch batch_norm (training statistics) in fp64, a
    hand-derived fixture, per-column mean 0 / variance 1 at eps = 0, a
    constant column gives beta, column permutation equivariance, the returned
    mean and biased variance against the statistics module."""
    import torch
    fails = []
    rng = np.random.Generator(np.random.PCG64(32))
    M, N = 41, 13
    A = rng.standard_normal((M, N)) * 3 + rng.standard_normal(N) * 4
    g = 1 + 0.3 * rng.standard_normal(N)
    b = 0.2 * rng.standard_normal(N)
    ref = torch.nn.functional.batch_norm(torch.from_numpy(A), None, None, torch.from_numpy(g), torch.from_numpy(b),
                                         training=True, eps=1e-5).numpy()
    y, mean, var = fn(A, g, b, 1e-5)
    y = np.asarray(y)
    _fail(fails, y.shape == ref.shape and np.allclose(y, ref, rtol=1e-12, atol=1e-12), "BN vs torch batch_norm")
    cols = A.T.tolist()
    _fail(fails, all(abs(mean[j] - statistics.fmean(cols[j])) < 1e-12 for j in range(N)), "BN mean")
    _fail(fails, all(abs(var[j] - statistics.pvariance(cols[j])) < 1e-10 * (1 + var[j]) for j in range(N)),
          "BN biased variance")
    gold = _load_golden("batchnorm_worked.txt")
    yg = np.asarray(fn(np.array([[1.0, 10], [3, 10], [5, 16]]), np.array([2.0, 1]), np.array([0.0, 0.5]), 0.0)[0])
    _fail(fails, np.allclose(yg, gold, rtol=0, atol=1e-14), "BN hand-derived fixture")
    yn = np.asarray(fn(A, np.ones(N), np.zeros(N), 0.0)[0])
    _fail(fails, np.all(np.abs(yn.mean(axis=0)) < 1e-12), "BN columns have mean 0 at eps = 0")
    _fail(fails, all(abs(statistics.pvariance(c) - 1) < 1e-9 for c in yn.T.tolist()), "BN columns have variance 1")
    Ac = A.copy()
    Ac[:, 4] = 2.5
    yc = np.asarray(fn(Ac, g, b, 1e-5)[0])
    _fail(fails, np.all(yc[:, 4] == b[4]), "BN constant column gives beta")
    perm = rng.permutation(N)
    yp = np.asarray(fn(A[:, perm], g[perm], b[perm], 1e-5)[0])
    _fail(fails, np.allclose(yp, y[:, perm], rtol=1e-13, atol=1e-13), "BN column permutation")
    return fails


def check_stitch(st) -> list:
    fails = []
    rng = np.random.Generator(np.random.PCG64(16))
    # row [0, c]: y = [b, c^3 + b] -> [1/(1+e^{c^3}), e^{c^3}/(1+e^{c^3})]
    for c, b in ((0.7, 0.4), (-1.3, -0.9)):
        y = np.asarray(st(np.array([[0.0, c]]), np.array([b])))[0]
        p1 = 1 / (1 + math.exp(-(c ** 3)))
        _fail(fails, abs(y[1] - p1) < 1e-15 and abs(y[0] - (1 - p1)) < 1e-15,
              f"stitch two-element closed form c={c}")
    # the cube keeps its sign: A = [-1, 1] -> y = [-1+b, 1+b]
    y = np.asarray(st(np.array([[-1.0, 1.0]]), np.array([0.5])))[0]
    _fail(fails, abs(y[0] - 1 / (1 + math.e ** 2)) < 1e-15, "stitch cube sign")
    # the row bias is a per-row shift: the result equals the zero-bias one
    A = rng.standard_normal((5, 32)) * 2
    b = rng.random(5) * 2 - 1
    y1 = np.asarray(st(A, b))
    y0 = np.asarray(st(A, np.zeros(5)))
    _fail(fails, np.allclose(y1, y0, rtol=1e-12, atol=1e-300), "stitch row-bias shift invariance")
    _fail(fails, np.all(np.abs(y1.sum(axis=1) - 1) < 1e-12), "stitch row sums")
    # brute force on a tiny case with Python floats
    A = rng.standard_normal((3, 5))
    b = rng.random(3)
    ref = np.zeros_like(A)
    for i in range(3):
        yv = [float(A[i, j]) ** 3 + float(b[i]) for j in range(5)]
        m = max(yv)
        e = [math.exp(v - m) for v in yv]
        s = math.fsum(e)
        ref[i] = [v / s for v in e]
    _fail(fails, np.allclose(np.asarray(st(A, b)), ref, rtol=1e-13, atol=1e-16), "stitch brute force")
    return fails


def check_stitch_powadd(fn) -> list:
    """out = softmax_row(A + w[col]^p): closed forms, invariants, brute force."""
    fails = []
    rng = np.random.Generator(np.random.PCG64(18))
    A = rng.standard_normal((4, 9))
    w = rng.random(9) * 1.5 + 0.5
    # p = 0: every power is 1, a shift of every row: the plain row softmax
    e = np.exp(A - A.max(axis=1, keepdims=True))
    ref = e / e.sum(axis=1, keepdims=True)
    _fail(fails, np.allclose(np.asarray(fn(A, w, 0.0)), ref, rtol=1e-13, atol=1e-300), "powadd p=0 is softmax(A)")
    # w = 1: 1^p = 1 for any p
    ones = np.ones(9)
    _fail(fails, np.allclose(np.asarray(fn(A, ones, 2.7)), ref, rtol=1e-13, atol=1e-300), "powadd w=1")
    # two-element row [a0, a1] with [w0, w1], p = 2: sigmoid of the difference
    a0, a1, w0, w1 = 0.3, -0.2, 1.5, 0.5
    y = np.asarray(fn(np.array([[a0, a1]]), np.array([w0, w1]), 2.0))[0]
    d = (a1 + w1 * w1) - (a0 + w0 * w0)
    p1 = 1 / (1 + math.exp(-d))
    _fail(fails, abs(y[1] - p1) < 1e-15 and abs(y[0] - (1 - p1)) < 1e-15, "powadd two-element closed form")
    # the power broadcasts along the rows (one value per column): A = 0 gives
    # the softmax of w^p in every row
    z = np.asarray(fn(np.zeros((3, 9)), w, 1.5))
    pw = [float(x) ** 1.5 for x in w]
    m = max(pw)
    ez = [math.exp(v - m) for v in pw]
    sz = math.fsum(ez)
    _fail(fails, all(np.allclose(z[i], [v / sz for v in ez], rtol=1e-13) for i in range(3)),
          "powadd column broadcast")
    # brute force with Python floats (math.pow, math.fsum), non-integer p
    B = rng.standard_normal((3, 6))
    v = rng.random(6) + 0.25
    p = 2.5
    bf = np.zeros_like(B)
    for i in range(3):
        yv = [float(B[i, j]) + math.pow(float(v[j]), p) for j in range(6)]
        mm = max(yv)
        ev = [math.exp(t - mm) for t in yv]
        ss = math.fsum(ev)
        bf[i] = [t / ss for t in ev]
    _fail(fails, np.allclose(np.asarray(fn(B, v, p)), bf, rtol=1e-13, atol=1e-16), "powadd brute force")
    out = np.asarray(fn(B, v, p))
    _fail(fails, np.all(np.abs(out.sum(axis=1) - 1) < 1e-12), "powadd row sums")
    # rows= selects rows of the full result
    rws = np.array([2, 0])
    _fail(fails, np.array_equal(np.asarray(fn(B, v, p, rows=rws)), out[rws]), "powadd rows= sampling")
    return fails
