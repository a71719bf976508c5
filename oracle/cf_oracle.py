"""Plain, slow, fp64 CPU oracle for the fused GEMM + row-reduce/broadcast path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path; the only thing both sides share is the seeded
input generator, which holds none of the method's arithmetic.

What is computed, and where it is defined
-----------------------------------------
The pages describe *exact* fusion: the fused kernel must reach the result of
the unfused operator chain (the fusion keeps the semantics of the unfused
operators: ComFuse, Fusion Spec IR, Eq. (10); ownership legality: sass2mlir
"Kernel fusion", section "Epilogue fusion - the core technique").  So the oracle is the unfused chain
written out in float64 on the same (bf16 / fp32) input values:

* MatMul      P = X . W                       (ComFuse, Eq. (6) notation)
* Stage 1     x = alpha * P + bias            (ComFuse, Stage-Stream Execution
                                               Model, Fig. 3: x = alpha*Acc+Bias)
* activation  g = GELU_tanh(x) or g = x       (a unary compute node, ComFuse,
                                               Fusion Spec IR mapping Phi)
* reduction   LayerNorm / RMSNorm / Softmax as "reduce over the inputs,
              normalise the original values" (ComFuse, nested Fusion Spec IR
              at reductions, which names all three patterns)
* stitched    y = A^3 + b[row]; rowwise softmax (AStitch, "Adaptive thread
              mapping": row reductions on 750000x32 and 64x30000)

Pages cited (full titles):
  ComFuse  -- "ComFuse: Fusing Complex Memory-Intensive Subgraphs with
              Compute-Intensive Kernels For Modern GPU Architectures"
  AStitch  -- "AStitch: enabling a new multi-dimensional optimization space for
              memory-intensive ML training and inference on modern SIMT
              architectures"
  sass2mlir -- the sass2mlir "kernel fusion" page ("Two answers to the same
              idle GPU": CUDA graphs, then "How we fuse kernels")

Readings taken where the pages are silent:
  * LayerNorm variance is the biased one (divide by N), eps inside the square
    root, gamma/beta applied after normalising; with GELU the norm is taken
    over the post-GELU values.
  * RMSNorm divides each value by sqrt(mean of the squares + eps) with no mean
    subtraction (the usual definition, Zhang & Sennrich 2019); gamma scales
    after normalising and beta, when given, is added last.
  * Residual add + norm: the residual R is added after the activation node
    and before the reduction (the "add & norm" of a transformer block).
  * B2BGEMM: O = S . W2 with S = F(alpha * X.W1 + b1) held in bf16 -- the
    dtype of the intermediate tensor the unfused chain would materialise
    (the tensor cores consume bf16 operands); F is GELU(tanh), the row
    softmax over N1 or the row LayerNorm over N1 (gamma1, beta1 per column).
  * Masked softmax: a causal mask keeps element (i, j) of the scaled scores
    iff j <= i + offset (masked elements are -inf before the softmax); a row
    with no kept element is all zeros.
  * Softmax scale multiplies the accumulator before max/exp; an optional bias
    is added after scaling.  Exponent base e.
  * GELU is the tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
  * pow(A, 3) is the real cube with its sign (A*A*A).
  * Stitched add + LayerNorm: x = A + R (R optional), LayerNorm over each
    row as above, gamma/beta indexed by column.
  * Stitched power -> broadcast -> add -> softmax: y = A + w[col]^p with w > 0
    (the real power function w^p = exp(p ln w)), then the row softmax; the
    power of each column is a one-to-many value (AStitch's power -> broadcast
    -> add example, "What people did before").
  * Stitched BatchNorm (training-mode statistics): per column j the mean and
    the biased variance over all rows; y = (A - mean_j) / sqrt(var_j + eps)
    * gamma_j + beta_j.  The column statistic is a one-to-many dependency
    over every row (AStitch, "Four stitching schemes": Regional when one
    block holds all rows of its columns, Global otherwise).

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, invariants, brute force on tiny inputs and library routines.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "gemm",
    "gemm_naive",
    "gelu_tanh",
    "layernorm_rows",
    "rmsnorm_rows",
    "softmax_rows",
    "gemm_bias_rownorm",
    "gemm_bias_rmsnorm",
    "gemm_bias_residual_norm",
    "gemm_rowsoftmax_causal",
    "b2b_gemm",
    "stitch_add_layernorm",
    "stitch_batchnorm",
    "gemm_rowsoftmax",
    "stitch_rowreduce_broadcast",
    "stitch_powadd_softmax",
    "ROW_CHUNK",
]

# Row chunk used to bound the oracle's memory on the large configurations.
# Chunking over rows changes nothing: every row is computed independently.
ROW_CHUNK = 1024

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_GELU_CUBIC = 0.044715


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def gemm(X, W) -> np.ndarray:
    """P = X . W in float64 (ComFuse, Eq. (6): X in R^{MxK}, W in R^{KxN}).

    bf16 inputs widen exactly to float64 and every bf16 x bf16 product is
    exact in float64, so the only rounding is the float64 summation.
    """
    X = _f64(X)
    W = _f64(W)
    if X.ndim != 2 or W.ndim != 2 or X.shape[1] != W.shape[0]:
        raise ValueError(f"gemm: incompatible shapes {X.shape} x {W.shape}")
    return X @ W


def gemm_naive(X, W) -> np.ndarray:
    """Triple-loop MatMul, pure Python.  For tiny inputs only (pins gemm)."""
    X = _f64(X)
    W = _f64(W)
    M, K = X.shape
    K2, N = W.shape
    if K != K2:
        raise ValueError("gemm_naive: inner dimensions differ")
    P = np.zeros((M, N), dtype=np.float64)
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += float(X[i, k]) * float(W[k, j])
            P[i, j] = s
    return P


def gelu_tanh(x) -> np.ndarray:
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = _f64(x)
    return 0.5 * x * (1.0 + np.tanh(_SQRT_2_OVER_PI * (x + _GELU_CUBIC * x * x * x)))


def layernorm_rows(g, gamma, beta, eps: float) -> np.ndarray:
    """LayerNorm over the last axis, two-pass.

    mean = (1/N) sum g;  var = (1/N) sum (g - mean)^2  (biased);
    y = (g - mean) / sqrt(var + eps) * gamma + beta.
    This is the pattern the ComFuse Fusion Spec IR nests at a Reduction
    node -- reduce over the inputs, then normalise the original values: the first
    reduction (mean) feeds the second (variance), whose statistic is then
    broadcast back over the row together with the bypassed values.
    """
    g = _f64(g)
    mean = g.mean(axis=-1, keepdims=True)
    d = g - mean
    var = (d * d).mean(axis=-1, keepdims=True)
    return d / np.sqrt(var + float(eps)) * _f64(gamma) + _f64(beta)


def rmsnorm_rows(g, gamma, beta, eps: float) -> np.ndarray:
    """y = g / sqrt(mean(g^2) + eps) * gamma (+ beta), each row of g.

    RMSNorm as a nested stage DAG (ComFuse, Fusion Spec IR): the reduction is
    the mean of the squares over the row; the PostOp rescales the original
    values.  ``beta`` may be None (no shift node).
    """
    g = _f64(g)
    ms = (g * g).mean(axis=-1, keepdims=True)
    y = g / np.sqrt(ms + float(eps)) * _f64(gamma)
    return y if beta is None else y + _f64(beta)


def softmax_rows(z) -> np.ndarray:
    """Row softmax: m = max z; e = exp(z - m); y = e / sum(e)."""
    z = _f64(z)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def _row_chunks(M: int, rows):
    if rows is None:
        for r0 in range(0, M, ROW_CHUNK):
            yield np.arange(r0, min(M, r0 + ROW_CHUNK))
    else:
        rows = np.asarray(rows, dtype=np.int64)
        for r0 in range(0, rows.size, ROW_CHUNK):
            yield rows[r0:r0 + ROW_CHUNK]


def gemm_bias_rownorm(X, W, bias, gamma, beta, *, alpha: float = 1.0,
                      eps: float = 1e-5, act: str = "none", rows=None) -> np.ndarray:
    """y = LayerNorm(act(alpha * X.W + bias)) * gamma + beta, row by row.

    ComFuse, Stage-Stream Execution Model, Fig. 3 (stage 1: x = alpha*Acc+Bias,
    mean; stage 2: x - mean, ...) with an optional GELU node between the
    bias add and the reductions.  ``rows`` selects a subset of output rows
    (every row is independent, so a sampled row is exact).
    ``bias`` may be None (no bias node).
    """
    if act not in ("none", "gelu_tanh"):
        raise ValueError(f"unknown activation {act!r}")
    X = np.asarray(X)
    M = X.shape[0]
    N = np.asarray(W).shape[1]
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N), dtype=np.float64)
    b = np.zeros(N) if bias is None else _f64(bias)
    o = 0
    for idx in _row_chunks(M, rows):
        x = float(alpha) * gemm(X[idx], W) + b
        g = gelu_tanh(x) if act == "gelu_tanh" else x
        out[o:o + idx.size] = layernorm_rows(g, gamma, beta, eps)
        o += idx.size
    return out


def gemm_bias_rmsnorm(X, W, bias, gamma, beta=None, *, alpha: float = 1.0,
                      eps: float = 1e-5, act: str = "none", rows=None) -> np.ndarray:
    """y = RMSNorm(act(alpha * X.W + bias)) * gamma (+ beta), row by row.

    The same stage-1 nodes as ``gemm_bias_rownorm`` (ComFuse, Stage-Stream
    Execution Model, Fig. 3: x = alpha*Acc+Bias, then the optional GELU node)
    followed by the RMSNorm reduction and PostOp.
    """
    if act not in ("none", "gelu_tanh"):
        raise ValueError(f"unknown activation {act!r}")
    X = np.asarray(X)
    M = X.shape[0]
    N = np.asarray(W).shape[1]
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N), dtype=np.float64)
    b = np.zeros(N) if bias is None else _f64(bias)
    o = 0
    for idx in _row_chunks(M, rows):
        x = float(alpha) * gemm(X[idx], W) + b
        g = gelu_tanh(x) if act == "gelu_tanh" else x
        out[o:o + idx.size] = rmsnorm_rows(g, gamma, beta, eps)
        o += idx.size
    return out


def gemm_bias_residual_norm(X, W, bias, R, gamma, beta, *, alpha: float = 1.0, eps: float = 1e-5,
                            act: str = "none", norm: str = "layer", rows=None) -> np.ndarray:
    """y = Norm(act(alpha * X.W + bias) + R) * gamma (+ beta), row by row.

    sass2mlir, "Epilogue fusion - the core technique": activation, norm and
    residual add run on the accumulator in the producer's epilogue.  The
    residual R [M, N] is one more elementwise node before the reduction
    (ComFuse, Stage-Stream Execution Model: stage-1 nodes, then the row
    reduction).  norm is "layer" (LayerNorm) or "rms" (RMSNorm; beta may be
    None there).
    """
    if act not in ("none", "gelu_tanh"):
        raise ValueError(f"unknown activation {act!r}")
    if norm not in ("layer", "rms"):
        raise ValueError(f"unknown norm {norm!r}")
    X = np.asarray(X)
    R = np.asarray(R)
    M = X.shape[0]
    N = np.asarray(W).shape[1]
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N), dtype=np.float64)
    b = np.zeros(N) if bias is None else _f64(bias)
    o = 0
    for idx in _row_chunks(M, rows):
        x = float(alpha) * gemm(X[idx], W) + b
        g = (gelu_tanh(x) if act == "gelu_tanh" else x) + _f64(R[idx])
        out[o:o + idx.size] = (layernorm_rows(g, gamma, beta, eps) if norm == "layer"
                               else rmsnorm_rows(g, gamma, beta, eps))
        o += idx.size
    return out


def gemm_rowsoftmax(X, W, *, scale: float, bias=None, rows=None) -> np.ndarray:
    """y = softmax(scale * X.W (+ bias)) over each row."""
    X = np.asarray(X)
    M = X.shape[0]
    N = np.asarray(W).shape[1]
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N), dtype=np.float64)
    o = 0
    for idx in _row_chunks(M, rows):
        z = float(scale) * gemm(X[idx], W)
        if bias is not None:
            z = z + _f64(bias)
        out[o:o + idx.size] = softmax_rows(z)
        o += idx.size
    return out


def gemm_rowsoftmax_causal(X, W, *, scale: float, offset: int, bias=None, rows=None) -> np.ndarray:
    """y = softmax(mask(scale * X.W (+ bias))) over each row, where the mask
    keeps column j of row i iff j <= i + offset; a fully masked row is 0.

    A masked reduction node ahead of Softmax's nested stage DAG (ComFuse,
    Fusion Spec IR): masked elements take no part in the max or the sum and
    are 0 in the output.
    """
    X = np.asarray(X)
    M = X.shape[0]
    N = np.asarray(W).shape[1]
    idx_all = np.arange(M) if rows is None else np.asarray(rows)
    out = np.zeros((idx_all.size, N), dtype=np.float64)
    o = 0
    for idx in _row_chunks(M, rows):
        z = float(scale) * gemm(X[idx], W)
        if bias is not None:
            z = z + _f64(bias)
        keep = np.arange(N)[None, :] <= (idx[:, None] + int(offset))
        for r in range(idx.size):
            if keep[r].any():
                out[o + r, keep[r]] = softmax_rows(z[r, keep[r]][None, :])[0]
        o += idx.size
    return out


def b2b_gemm(X, W1, W2, *, op: str, alpha: float = 1.0, b1=None, rows=None, gamma1=None, beta1=None,
             eps: float = 1e-5) -> np.ndarray:
    """O = bf16(F(alpha * X.W1 + b1)) . W2, F = GELU_tanh, the row softmax or
    the row LayerNorm (with gamma1, beta1 over the N1 columns).

    ComFuse, B2BGEMM (Eqs. 3-7): MatMul_1, the epilogue F giving S_tile
    (Eq. 3), MatMul_2 over the intermediate dimension N1 (Eqs. 4-5).  The
    intermediate S is rounded to bf16 (round to nearest even), the precision
    of the tensor the unfused chain stores between the two GEMMs.
    """
    if op not in ("softmax", "gelu_tanh", "layernorm"):
        raise ValueError(f"unknown op {op!r}")
    X = np.asarray(X)
    M = X.shape[0]
    N2 = np.asarray(W2).shape[1]
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N2), dtype=np.float64)
    b = 0.0 if b1 is None else _f64(b1)
    o = 0
    for idx in _row_chunks(M, rows):
        z = float(alpha) * gemm(X[idx], W1) + b
        if op == "softmax":
            S = softmax_rows(z)
        elif op == "gelu_tanh":
            S = gelu_tanh(z)
        else:
            S = layernorm_rows(z, gamma1, beta1, eps)
        S = _round_bf16(S)
        out[o:o + idx.size] = gemm(S, W2)
        o += idx.size
    return out


def _round_bf16(a) -> np.ndarray:
    """Nearest bf16 value (ties to even) of each element, via float32."""
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def stitch_add_layernorm(A, R, gamma, beta, eps: float, rows=None) -> np.ndarray:
    """out = LayerNorm(A + R) * gamma + beta over each row (R may be None).

    AStitch, "Four stitching schemes": an elementwise producer (Local), two
    reductions over the row (mean, then the variance around it) and their
    broadcast back, with column parameters shared by every row (a
    one-to-many dependency: Regional).
    """
    A = np.asarray(A)
    M, N = A.shape
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N), dtype=np.float64)
    o = 0
    for idx in _row_chunks(M, rows):
        x = _f64(A[idx])
        if R is not None:
            x = x + _f64(np.asarray(R)[idx])
        out[o:o + idx.size] = layernorm_rows(x, gamma, beta, eps)
        o += idx.size
    return out


def stitch_batchnorm(A, gamma, beta, eps: float):
    """BatchNorm over the rows of A [rows, cols] with batch statistics.

    mean_j = (1/rows) sum_i A_ij;  var_j = (1/rows) sum_i (A_ij - mean_j)^2;
    out_ij = (A_ij - mean_j) / sqrt(var_j + eps) * gamma_j + beta_j.
    Returns (out, mean, var).  Every output depends on every row of its
    column: the reduction runs along the other axis from the row reductions
    (AStitch, "Four stitching schemes", column reduction -> broadcast).
    """
    A = _f64(A)
    mean = A.mean(axis=0)
    d = A - mean
    var = (d * d).mean(axis=0)
    return d / np.sqrt(var + float(eps)) * _f64(gamma) + _f64(beta), mean, var


def stitch_rowreduce_broadcast(A, row_bias, rows=None) -> np.ndarray:
    """Stitched memory-intensive subgraph (AStitch, "Adaptive thread mapping"):

    y = A*A*A + b[row]  (elementwise power, then a broadcast row bias);
    m = rowmax(y); s = rowsum(exp(y - m)); out = exp(y - m) / s.
    """
    A = np.asarray(A)
    b = np.asarray(row_bias)
    M, N = A.shape
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N), dtype=np.float64)
    o = 0
    for idx in _row_chunks(M, rows):
        a = _f64(A[idx])
        y = a * a * a + _f64(b[idx])[:, None]
        out[o:o + idx.size] = softmax_rows(y)
        o += idx.size
    return out


def stitch_powadd_softmax(A, w, p: float, rows=None) -> np.ndarray:
    """Stitched subgraph with both one-to-many dependencies (AStitch, "What
    people did before": an expensive element-wise power feeding a broadcast
    and an add; "Four stitching schemes": the reduction feeding consumers):

    y = A + w[col] ** p   (w > 0: the real power w^p = exp(p ln w));
    m = rowmax(y); s = rowsum(exp(y - m)); out = exp(y - m) / s.
    """
    A = np.asarray(A)
    w = _f64(w)
    if np.any(w <= 0):
        raise ValueError("stitch_powadd_softmax: w must be positive")
    pw = w ** float(p)
    M, N = A.shape
    out_rows = M if rows is None else len(rows)
    out = np.empty((out_rows, N), dtype=np.float64)
    o = 0
    for idx in _row_chunks(M, rows):
        y = _f64(A[idx]) + pw[None, :]
        out[o:o + idx.size] = softmax_rows(y)
        o += idx.size
    return out
