"""The fp64 oracle against what the mathematics fixes (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


def test_gemm_pinned():
    assert pins.check_gemm(oracle.gemm) == []


def test_gemm_naive_pinned():
    assert pins.check_gemm(oracle.gemm_naive) == []


def test_gemm_agrees_with_naive_triple_loop():
    rng = np.random.Generator(np.random.PCG64(1))
    for M, K, N in [(3, 7, 5), (17, 9, 11)]:
        X = np.round(rng.standard_normal((M, K)) * 128) / 128
        W = np.round(rng.standard_normal((K, N)) * 128) / 128
        np.testing.assert_allclose(oracle.gemm(X, W), oracle.gemm_naive(X, W), rtol=1e-12, atol=1e-13)


def test_gelu_pinned():
    assert pins.check_gelu(oracle.gelu_tanh) == []


def test_layernorm_pinned():
    assert pins.check_layernorm(oracle.layernorm_rows) == []


def test_rmsnorm_pinned():
    assert pins.check_rmsnorm(oracle.rmsnorm_rows) == []


def test_rmsnorm_composition_pinned():
    assert pins.check_rmsnorm_composition(oracle.gemm_bias_rmsnorm) == []


def test_residual_norm_pinned():
    assert pins.check_residual_norm(oracle.gemm_bias_residual_norm) == []


def test_softmax_pinned():
    assert pins.check_softmax(oracle.softmax_rows) == []


def test_rownorm_composition_pinned():
    assert pins.check_rownorm_composition(oracle.gemm_bias_rownorm) == []


def test_softmax_composition_pinned():
    assert pins.check_softmax_composition(oracle.gemm_rowsoftmax) == []


def test_softmax_causal_pinned():
    assert pins.check_softmax_causal(oracle.gemm_rowsoftmax_causal) == []


def test_b2b_pinned():
    assert pins.check_b2b(oracle.b2b_gemm) == []


def test_stitch_pinned():
    assert pins.check_stitch(oracle.stitch_rowreduce_broadcast) == []


def test_rownorm_gemm_matches_naive_composition_tiny():
    """The composed oracle with its GEMM replaced by the triple loop."""
    rng = np.random.Generator(np.random.PCG64(2))
    M, K, N = 4, 8, 6
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N))
    bias = rng.standard_normal(N)
    gam = rng.standard_normal(N)
    bet = rng.standard_normal(N)
    x = oracle.gemm_naive(X, W) + bias
    want = oracle.layernorm_rows(oracle.gelu_tanh(x), gam, bet, 1e-5)
    got = oracle.gemm_bias_rownorm(X, W, bias, gam, bet, eps=1e-5, act="gelu_tanh")
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_layernorm_unit_variance_at_config_scale():
    """At the FFN-sized workload's scale (row variance ~1.6e-4) eps=1e-5 pulls the
    variance of the normalised row to s2/(s2+eps) ~ 0.94; with eps=0 it is 1."""
    from memory_fusion_gb300.inputs import gemm_inputs
    d = gemm_inputs(8, 256, 512, 7, x_std=1 / np.sqrt(512), w_std=1 / np.sqrt(512),
                    bias_std=0.02, gamma_std=None, beta_std=None)
    N = 256
    y = oracle.gemm_bias_rownorm(d["X"], d["W"], d["bias"], np.ones(N), np.zeros(N),
                                 eps=0.0, act="gelu_tanh")
    assert np.all(np.abs(y.mean(1)) < 1e-9)
    assert np.all(np.abs(y.var(1) - 1) < 1e-9)


@pytest.mark.parametrize("rows", [None, [0, 5, 1]])
def test_row_chunking_is_transparent(rows, monkeypatch):
    from oracle import cf_oracle
    rng = np.random.Generator(np.random.PCG64(3))
    X = rng.standard_normal((7, 16))
    W = rng.standard_normal((16, 12))
    b = rng.standard_normal(12)
    full = cf_oracle.gemm_bias_rownorm(X, W, b, np.ones(12), np.zeros(12), rows=rows)
    monkeypatch.setattr(cf_oracle, "ROW_CHUNK", 2)
    chunked = cf_oracle.gemm_bias_rownorm(X, W, b, np.ones(12), np.zeros(12), rows=rows)
    np.testing.assert_allclose(full, chunked, rtol=1e-13, atol=1e-14)  # BLAS blocking may differ by 1 ulp


def test_stitch_add_layernorm_pinned():
    assert pins.check_stitch_add_layernorm(oracle.stitch_add_layernorm) == []


def test_stitch_batchnorm_pinned():
    assert pins.check_stitch_batchnorm(oracle.stitch_batchnorm) == []


def test_b2b_layernorm_fold_identity():
    """The stream kernel's one-pass LayerNorm rests on LayerNorm being affine
    in a row once its mean and rstd are fixed: for any shift mu0,
    LN(z) . W2 = rstd ((z - mu0) gamma) . W2 - rstd (mu - mu0) gamma^T W2 + beta^T W2.
    Checked in fp64 against the oracle's LayerNorm (before any bf16
    rounding) with mu0 the mean of each row's first 256 columns, on rows whose
    mean is far from 0 and whose first chunk is far from the row's mean."""
    rng = np.random.Generator(np.random.PCG64(31))
    M, N1, N2 = 8, 1024, 64
    z = rng.standard_normal((M, N1)) + 30.0 + 5.0 * np.linspace(-1.0, 1.0, N1)
    gamma = 1.0 + 0.1 * rng.standard_normal(N1)
    beta = 0.1 * rng.standard_normal(N1)
    W2 = rng.standard_normal((N1, N2))
    direct = oracle.layernorm_rows(z, gamma, beta, 1e-5) @ W2
    mu = z.mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(((z - mu) ** 2).mean(axis=1, keepdims=True) + 1e-5)
    mu0 = z[:, :256].mean(axis=1, keepdims=True)
    folded = rstd * (((z - mu0) * gamma) @ W2) - rstd * (mu - mu0) * (gamma @ W2) + beta @ W2
    np.testing.assert_allclose(folded, direct, rtol=1e-10, atol=1e-9 * np.abs(direct).max())


def test_stitch_powadd_pinned():
    assert pins.check_stitch_powadd(oracle.stitch_powadd_softmax) == []


def test_stitch_powadd_rejects_nonpositive_base():
    with pytest.raises(ValueError):
        oracle.stitch_powadd_softmax(np.zeros((1, 2)), np.array([1.0, 0.0]), 2.0)
