"""Plant plausible mistakes in copies of the oracle and check a pin catches each.

The mistakes live here, on the CPU, in throw-away lambdas; the oracle itself
is untouched.  Each mutant must fail at least one pin in ``oracle_pins``.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import cf_oracle
from tests import oracle_pins as pins

S = math.sqrt(2 / math.pi)


def _ln(g, gamma, beta, eps, *, ddof=0, eps_out=False, use_beta=True, center_out=True,
        gamma_first=False, var_about_zero=False):
    g = np.asarray(g, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    if gamma_first:
        g = g * gamma
    mean = g.mean(-1, keepdims=True)
    d = g - mean
    if var_about_zero:
        var = (g * g).mean(-1, keepdims=True)
    else:
        var = (d * d).sum(-1, keepdims=True) / (g.shape[-1] - ddof)
    den = (np.sqrt(var) + eps) if eps_out else np.sqrt(var + eps)
    y = (d if center_out else g) / den
    if not gamma_first:
        y = y * gamma
    return y + (beta if use_beta else 0.0)


LN_MUTANTS = {
    "unbiased variance": lambda g, ga, be, e: _ln(g, ga, be, e, ddof=1),
    "eps outside sqrt": lambda g, ga, be, e: _ln(g, ga, be, e, eps_out=True),
    "beta dropped": lambda g, ga, be, e: _ln(g, ga, be, e, use_beta=False),
    "mean not subtracted": lambda g, ga, be, e: _ln(g, ga, be, e, center_out=False),
    "gamma before normalising": lambda g, ga, be, e: _ln(g, ga, be, e, gamma_first=True),
    "variance about zero": lambda g, ga, be, e: _ln(g, ga, be, e, var_about_zero=True),
}


def _rms(g, gamma, beta, eps, *, center=False, eps_out=False, use_sum=False, beta_inside=False,
         gamma_first=False):
    g = np.asarray(g, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    b = 0.0 if beta is None else np.asarray(beta, dtype=np.float64)
    if beta_inside:
        g = g + b
    if gamma_first:
        g = g * gamma
    c = g - g.mean(-1, keepdims=True) if center else g
    ms = (c * c).sum(-1, keepdims=True) if use_sum else (c * c).mean(-1, keepdims=True)
    den = (np.sqrt(ms) + eps) if eps_out else np.sqrt(ms + eps)
    y = c / den
    if not gamma_first:
        y = y * gamma
    return y if beta_inside else y + b


RMS_MUTANTS = {
    "mean subtracted": lambda g, ga, be, e: _rms(g, ga, be, e, center=True),
    "eps outside sqrt": lambda g, ga, be, e: _rms(g, ga, be, e, eps_out=True),
    "sum of squares": lambda g, ga, be, e: _rms(g, ga, be, e, use_sum=True),
    "beta before normalising": lambda g, ga, be, e: _rms(g, ga, be, e, beta_inside=True),
    "gamma before normalising": lambda g, ga, be, e: _rms(g, ga, be, e, gamma_first=True),
}


def _sm(z, *, sub_max=True, base=math.e, by_max=False):
    z = np.asarray(z, dtype=np.float64)
    m = z.max(-1, keepdims=True) if sub_max else 0.0
    e = np.power(base, z - m)
    return e / (e.max(-1, keepdims=True) if by_max else e.sum(-1, keepdims=True))


SM_MUTANTS = {
    "no max subtraction": lambda z: _sm(z, sub_max=False),
    "base 2": lambda z: _sm(z, base=2.0),
    "divide by max": lambda z: _sm(z, by_max=True),
    "softmax over columns": lambda z: (lambda zz: np.exp(zz - zz.max(0)) / np.exp(zz - zz.max(0)).sum(0))(np.asarray(z, dtype=np.float64)),
}

GELU_MUTANTS = {
    "cubic coefficient": lambda x: 0.5 * x * (1 + np.tanh(S * (x + 0.0447 * x ** 3))),
    "sqrt(2/pi) dropped": lambda x: 0.5 * x * (1 + np.tanh(x + 0.044715 * x ** 3)),
    "sigmoid form": lambda x: x / (1 + np.exp(-1.702 * x)),
    "missing half": lambda x: x * (1 + np.tanh(S * (x + 0.044715 * x ** 3))),
    "erf form": lambda x: 0.5 * x * (1 + np.vectorize(math.erf)(np.asarray(x) / math.sqrt(2))),
}

GEMM_MUTANTS = {
    "transposed W": lambda X, W: np.asarray(X) @ np.asarray(W).T if np.asarray(W).shape[0] == np.asarray(W).shape[1] else (np.asarray(X) @ np.asarray(W)).T,
    "dropped last k term": lambda X, W: np.asarray(X, float)[:, :-1] @ np.asarray(W, float)[:-1],
    "fp32 accumulation": lambda X, W: (np.asarray(X, np.float32) @ np.asarray(W, np.float32)).astype(np.float64) + 1e-9,
}


def _rownorm(X, W, bias, gamma, beta, *, alpha=1.0, eps=1e-5, act="none", rows=None,
             order="ok"):
    X = np.asarray(X, float)
    if rows is not None:
        X = X[rows]
    P = X @ np.asarray(W, float)
    b = 0.0 if bias is None else np.asarray(bias, float)
    x = alpha * (P + b) if order == "bias before alpha" else alpha * P + b
    if order == "gelu after norm":
        y = oracle.layernorm_rows(x, gamma, beta, eps)
        return oracle.gelu_tanh(y) if act == "gelu_tanh" else y
    g = oracle.gelu_tanh(x) if act == "gelu_tanh" else x
    if order == "bias after gelu":
        g = (oracle.gelu_tanh(alpha * P) if act == "gelu_tanh" else alpha * P) + b
    return oracle.layernorm_rows(g, gamma, beta, eps)


ROWNORM_MUTANTS = {
    k: (lambda kk: (lambda *a, **kw: _rownorm(*a, order=kk, **kw)))(k)
    for k in ("bias before alpha", "gelu after norm", "bias after gelu")
}


def _softmax_fused(X, W, *, scale, bias=None, rows=None, mistake):
    X = np.asarray(X, float)
    if rows is not None:
        X = X[rows]
    z = X @ np.asarray(W, float)
    if mistake == "scale after bias" and bias is not None:
        z = scale * (z + np.asarray(bias))
    elif mistake == "bias ignored":
        z = scale * z
    elif mistake == "scale dropped":
        z = z + (0 if bias is None else np.asarray(bias))
    else:
        z = scale * z + (0 if bias is None else np.asarray(bias))
    return oracle.softmax_rows(z)


SOFTMAX_FUSED_MUTANTS = {k: (lambda kk: (lambda *a, **kw: _softmax_fused(*a, mistake=kk, **kw)))(k)
                         for k in ("scale after bias", "bias ignored", "scale dropped")}


def _stitch(A, b, rows=None, *, mistake):
    A = np.asarray(A, float)
    b = np.asarray(b, float)
    if mistake == "square":
        y = A * A + b[:, None]
    elif mistake == "abs cube":
        y = np.abs(A) ** 3 + b[:, None]
    elif mistake == "bias multiplies":
        y = A ** 3 * b[:, None]
    else:
        y = A ** 3 + b[None, :A.shape[1]] if A.shape[1] == b.shape[0] else A ** 3 - b[:, None] * A
    return oracle.softmax_rows(y)


STITCH_MUTANTS = {k: (lambda kk: (lambda A, b, rows=None: _stitch(A, b, rows, mistake=kk)))(k)
                  for k in ("square", "abs cube", "bias multiplies", "bias per column")}


@pytest.mark.parametrize("name", sorted(LN_MUTANTS))
def test_layernorm_mutant_caught(name):
    assert pins.check_layernorm(LN_MUTANTS[name]), name


@pytest.mark.parametrize("name", sorted(RMS_MUTANTS))
def test_rmsnorm_mutant_caught(name):
    with np.errstate(invalid="ignore", divide="ignore"):  # centring a 1-column row gives 0/0
        assert pins.check_rmsnorm(RMS_MUTANTS[name]), name


@pytest.mark.parametrize("name", sorted(SM_MUTANTS))
def test_softmax_mutant_caught(name):
    with np.errstate(over="ignore", invalid="ignore"):
        assert pins.check_softmax(SM_MUTANTS[name]), name


@pytest.mark.parametrize("name", sorted(GELU_MUTANTS))
def test_gelu_mutant_caught(name):
    assert pins.check_gelu(GELU_MUTANTS[name]), name


@pytest.mark.parametrize("name", sorted(GEMM_MUTANTS))
def test_gemm_mutant_caught(name):
    assert pins.check_gemm(GEMM_MUTANTS[name]), name


@pytest.mark.parametrize("name", sorted(ROWNORM_MUTANTS))
def test_rownorm_mutant_caught(name):
    assert pins.check_rownorm_composition(ROWNORM_MUTANTS[name]), name


@pytest.mark.parametrize("name", sorted(SOFTMAX_FUSED_MUTANTS))
def test_softmax_composition_mutant_caught(name):
    assert pins.check_softmax_composition(SOFTMAX_FUSED_MUTANTS[name]), name


def _residual(X, W, bias, R, gamma, beta, *, alpha=1.0, eps=1e-5, act="none", norm="layer", rows=None,
              mistake):
    X = np.asarray(X, float)
    R = np.asarray(R, float)
    if rows is not None:
        X, R = X[rows], R[rows]
    x = alpha * (X @ np.asarray(W, float)) + (0 if bias is None else np.asarray(bias))
    if mistake == "residual before GELU":
        g = oracle.gelu_tanh(x + R) if act == "gelu_tanh" else x + R
    elif mistake == "residual after norm":
        g = oracle.gelu_tanh(x) if act == "gelu_tanh" else x
        y = oracle.layernorm_rows(g, gamma, beta, eps) if norm == "layer" else oracle.rmsnorm_rows(g, gamma, beta, eps)
        return y + R
    elif mistake == "residual scaled by alpha":
        g = alpha * R + (oracle.gelu_tanh(x) if act == "gelu_tanh" else x)
    else:
        g = (oracle.gelu_tanh(x) if act == "gelu_tanh" else x) + R.T[:R.shape[0], :R.shape[1]] if R.shape[0] == R.shape[1] else (oracle.gelu_tanh(x) if act == "gelu_tanh" else x) - R
    return oracle.layernorm_rows(g, gamma, beta, eps) if norm == "layer" else oracle.rmsnorm_rows(g, gamma, beta, eps)


RESIDUAL_MUTANTS = {k: (lambda kk: (lambda *a, **kw: _residual(*a, mistake=kk, **kw)))(k)
                    for k in ("residual before GELU", "residual after norm", "residual scaled by alpha",
                              "residual subtracted")}


@pytest.mark.parametrize("name", sorted(RESIDUAL_MUTANTS))
def test_residual_mutant_caught(name):
    assert pins.check_residual_norm(RESIDUAL_MUTANTS[name]), name


def _causal(X, W, *, scale, offset, bias=None, rows=None, mistake):
    X = np.asarray(X, float)
    M = X.shape[0]
    idx = np.arange(M) if rows is None else np.asarray(rows)
    z = scale * (X[idx] @ np.asarray(W, float)) + (0 if bias is None else np.asarray(bias))
    N = z.shape[1]
    if mistake == "strict inequality":
        keep = np.arange(N)[None, :] < idx[:, None] + offset
    elif mistake == "mask transposed":
        keep = np.arange(N)[None, :] >= idx[:, None] - offset
    else:
        keep = np.arange(N)[None, :] <= idx[:, None] + offset
    if mistake == "masked entries keep exp":
        e = np.exp(z - np.where(keep, z, -np.inf).max(1, keepdims=True).clip(-1e300))
        y = e / np.where(keep, e, 0).sum(1, keepdims=True)
        return np.nan_to_num(y)
    e = np.where(keep, np.exp(z - np.where(keep, z, -np.inf).max(1, keepdims=True).clip(-1e300)), 0.0)
    s = e.sum(1, keepdims=True)
    return np.divide(e, s, out=np.zeros_like(e), where=s > 0)


CAUSAL_MUTANTS = {k: (lambda kk: (lambda *a, **kw: _causal(*a, mistake=kk, **kw)))(k)
                  for k in ("strict inequality", "mask transposed", "masked entries keep exp")}


@pytest.mark.parametrize("name", sorted(CAUSAL_MUTANTS))
def test_causal_mutant_caught(name):
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        assert pins.check_softmax_causal(CAUSAL_MUTANTS[name]), name


def _b2b(X, W1, W2, *, op, alpha=1.0, b1=None, rows=None, gamma1=None, beta1=None, eps=1e-5, mistake):
    X = np.asarray(X, float)
    if rows is not None:
        X = X[rows]
    bias = 0 if (b1 is None or mistake == "b1 dropped") else np.asarray(b1)
    if mistake == "alpha after bias":
        z = alpha * (X @ np.asarray(W1, float) + bias)
    else:
        z = alpha * (X @ np.asarray(W1, float)) + bias
    if op == "softmax":
        S = oracle.softmax_rows(z.T).T if mistake == "softmax over columns" else oracle.softmax_rows(z)
    elif op == "layernorm":
        m = z.mean(axis=1, keepdims=True)
        dz = z - m
        n = z.shape[1] - (1 if mistake == "layernorm unbiased variance" else 0)
        S = dz / np.sqrt((dz * dz).sum(axis=1, keepdims=True) / n + eps) * np.asarray(gamma1) + np.asarray(beta1)
    else:
        S = oracle.gelu_tanh(z)
    if mistake == "no bf16 rounding":
        pass
    elif mistake == "fp16 rounding":
        S = S.astype(np.float16).astype(np.float64)
    elif mistake == "truncated to bf16":
        S = S.astype(np.float32).view(np.uint32)
        S = ((S >> 16) << 16).view(np.float32).astype(np.float64)  # truncation instead of rounding
    else:
        S = cf_oracle._round_bf16(S)
    if mistake == "W2 transposed" and np.asarray(W2).shape[0] == np.asarray(W2).shape[1]:
        return S @ np.asarray(W2, float).T
    return S @ np.asarray(W2, float)


B2B_MUTANTS = {k: (lambda kk: (lambda *a, **kw: _b2b(*a, mistake=kk, **kw)))(k)
               for k in ("no bf16 rounding", "fp16 rounding", "truncated to bf16", "b1 dropped", "alpha after bias",
                         "softmax over columns", "layernorm unbiased variance")}


@pytest.mark.parametrize("name", sorted(B2B_MUTANTS))
def test_b2b_mutant_caught(name):
    assert pins.check_b2b(B2B_MUTANTS[name]), name


def _add_ln(A, R, gamma, beta, eps, rows=None, *, mistake):
    A = np.asarray(A, float)
    x = A if R is None else (A - np.asarray(R, float) if mistake == "R subtracted" else A + np.asarray(R, float))
    if rows is not None:
        x = x[rows]
    ax = 0 if mistake == "normalised over columns" else -1
    mean = x.mean(axis=ax, keepdims=True)
    d = x - mean
    var = (d * d).sum(axis=ax, keepdims=True) / (x.shape[ax] - (1 if mistake == "unbiased variance" else 0))
    g, b = (beta, gamma) if mistake == "gamma and beta swapped" else (gamma, beta)
    return d / np.sqrt(var + eps) * np.asarray(g, float) + np.asarray(b, float)


ADD_LN_MUTANTS = {k: (lambda kk: (lambda *a, **kw: _add_ln(*a, mistake=kk, **kw)))(k)
                  for k in ("R subtracted", "normalised over columns", "unbiased variance", "gamma and beta swapped")}


@pytest.mark.parametrize("name", sorted(ADD_LN_MUTANTS))
def test_add_layernorm_mutant_caught(name):
    with np.errstate(divide="ignore", invalid="ignore"):
        assert pins.check_stitch_add_layernorm(ADD_LN_MUTANTS[name]), name


def _bn(A, gamma, beta, eps, *, mistake):
    A = np.asarray(A, float)
    ax = 1 if mistake == "normalised over rows" else 0
    mean = A.mean(axis=ax, keepdims=True)
    d = A - mean
    n = A.shape[ax]
    var = (d * d).sum(axis=ax, keepdims=True) / (n - 1 if mistake == "unbiased variance" else n)
    if mistake == "eps outside the root":
        y = d / (np.sqrt(var) + eps)
    else:
        y = d / np.sqrt(var + eps)
    if mistake == "gamma added":
        y = y + np.asarray(gamma, float) + np.asarray(beta, float)
    else:
        y = y * np.asarray(gamma, float) + np.asarray(beta, float)
    return y, mean.reshape(-1), var.reshape(-1)


BN_MUTANTS = {k: (lambda kk: (lambda *a, **kw: _bn(*a, mistake=kk, **kw)))(k)
              for k in ("normalised over rows", "unbiased variance", "eps outside the root", "gamma added")}


@pytest.mark.parametrize("name", sorted(BN_MUTANTS))
def test_batchnorm_mutant_caught(name):
    with np.errstate(divide="ignore", invalid="ignore"):
        assert pins.check_stitch_batchnorm(BN_MUTANTS[name]), name


@pytest.mark.parametrize("name", sorted(STITCH_MUTANTS))
def test_stitch_mutant_caught(name):
    with np.errstate(over="ignore", invalid="ignore"):
        assert pins.check_stitch(STITCH_MUTANTS[name]), name


def _powadd(A, w, p, rows=None, *, mistake):
    A = np.asarray(A, float)
    w = np.asarray(w, float)
    if rows is not None:
        A = A[np.asarray(rows)]
    if mistake == "power per row":          # broadcast along the wrong axis
        k = min(A.shape)
        y = A.copy()
        y[:k, :] += (w[:k] ** p)[:, None]
    elif mistake == "power multiplies":     # A * w^p instead of A + w^p
        y = A * (w ** p)[None, :]
    elif mistake == "base times exponent":  # w * p instead of w^p
        y = A + (w * p)[None, :]
    elif mistake == "exponent reciprocal":  # w^(1/p)
        y = A + (w ** (1.0 / p if p else 0.0))[None, :]
    elif mistake == "softmax over columns":
        y = A + (w ** p)[None, :]
        e = np.exp(y - y.max(axis=0, keepdims=True))
        return e / e.sum(axis=0, keepdims=True)
    else:
        raise ValueError(mistake)
    return oracle.softmax_rows(y)


POWADD_MUTANTS = {k: (lambda kk: (lambda A, w, p, rows=None: _powadd(A, w, p, rows, mistake=kk)))(k)
                  for k in ("power per row", "power multiplies", "base times exponent", "exponent reciprocal",
                            "softmax over columns")}


@pytest.mark.parametrize("name", sorted(POWADD_MUTANTS))
def test_powadd_mutant_caught(name):
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        assert pins.check_stitch_powadd(POWADD_MUTANTS[name]), name
