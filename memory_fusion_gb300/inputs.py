"""Seeded synthetic inputs, shared by the CUDA path's tests/bench and the oracle.

This module holds none of the method's arithmetic: it only draws random
numbers and rounds them to the storage type the workload names (bf16 by
round-to-nearest-even).  Both sides receive the very same values.

Recipe (one ``numpy.random.Generator(PCG64(seed))`` per workload, values drawn
as float64 normals / uniforms, scaled, cast to float32, then -- where the
workload stores bf16 -- rounded to bf16 with round-to-nearest-even; draws are
made in argument order):

* GEMM + row-norm workloads: X[M,K], W[K,N] (bf16, N(0, x_std), N(0, w_std));
  bias[N] ~ N(0, bias_std), gamma[N] ~ N(1, gamma_std), beta[N] ~ N(0,
  beta_std) (fp32).
* GEMM + softmax workloads: X, W as above; no bias unless asked.
* Stitched workload: A[rows, cols] ~ N(0, 2) fp32, then b[rows] ~ U(-1, 1)
  fp32; the generator is re-seeded for every shape.
* Stitched normalisation workloads: A[rows, cols] ~ N(0, 2) fp32, then (add
  + LayerNorm only) R[rows, cols] ~ N(0, 1), then gamma[cols] ~ N(1, 0.1),
  beta[cols] ~ N(0, 0.1) fp32.
* Back-to-back GEMM workloads: X[M,K], W1[K,N1], W2[N1,N2] (bf16, N(0,
  x_std), N(0, w1_std), N(0, w2_std)), then b1[N1] ~ N(0, b1_std) fp32 (not
  drawn when b1_std is None), then (LayerNorm epilogue) gamma1 ~ N(1, 0.1),
  beta1 ~ N(0, 0.1) [N1] fp32.

"N(0, s)" means standard deviation s throughout.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "round_to_bf16",
    "bf16_bits",
    "GemmWorkload",
    "StitchWorkload",
    "B2bWorkload",
    "StitchNormWorkload",
    "StitchPowWorkload",
    "stitch_norm_inputs",
    "powadd_inputs",
    "b2b_inputs",
    "WORKLOADS",
    "gemm_inputs",
    "stitch_inputs",
    "workload_inputs",
]


def round_to_bf16(a) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32.

    NaN/Inf are not produced by the generator; finite values only.
    """
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return bits.astype(np.uint32).view(np.float32).reshape(a.shape)


def bf16_bits(a_bf16_valued) -> np.ndarray:
    """uint16 bit patterns of float32 values that are exactly bf16."""
    a = np.ascontiguousarray(np.asarray(a_bf16_valued, dtype=np.float32))
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


@dataclass(frozen=True)
class GemmWorkload:
    name: str
    kind: str              # "rownorm" | "rmsnorm" | "softmax" | "softmax_causal"
    M: int
    N: int
    K: int
    seed: int
    x_std: float
    w_std: float
    bias_std: float | None = 0.0
    gamma_std: float = 0.0
    beta_std: float | None = 0.0
    act: str = "none"      # "none" | "gelu_tanh"
    eps: float = 1e-5
    resid_std: float | None = None  # a bf16 residual R [M, N] added before the norm
    mask_offset: int = 0   # softmax_causal: column j of row i kept iff j <= i + mask_offset
    alpha: float = 1.0
    scale: float = 1.0
    description: str = ""

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def unavoidable_bytes(self) -> int:
        """Inputs + final output, each once; no intermediate."""
        b = 2 * self.M * self.K + 2 * self.K * self.N + 2 * self.M * self.N
        if self.kind == "rownorm":
            b += 3 * 4 * self.N
        elif self.kind == "rmsnorm":
            b += (1 + (self.bias_std is not None) + (self.beta_std is not None)) * 4 * self.N
        if self.resid_std is not None:
            b += 2 * self.M * self.N
        return b


@dataclass(frozen=True)
class StitchWorkload:
    name: str
    rows: int
    cols: int
    seed: int
    description: str = ""

    @property
    def unavoidable_bytes(self) -> int:
        return 4 * self.rows * self.cols * 2 + 4 * self.rows


@dataclass(frozen=True)
class StitchNormWorkload:
    name: str
    kind: str              # "add_layernorm" | "batchnorm"
    rows: int
    cols: int
    seed: int
    eps: float = 1e-5
    description: str = ""

    @property
    def unavoidable_bytes(self) -> int:
        """Inputs and outputs once each: A (and R), out, gamma, beta (and the
        batch mean / variance BatchNorm returns)."""
        per = 12 if self.kind == "add_layernorm" else 8
        return per * self.rows * self.cols + (8 if self.kind == "add_layernorm" else 16) * self.cols


@dataclass(frozen=True)
class StitchPowWorkload:
    """out = softmax_row(A + w[col]^p): an expensive element-wise power of a
    column vector broadcast to every row, then the row reduction."""
    name: str
    rows: int
    cols: int
    seed: int
    p: float = 2.5
    description: str = ""

    @property
    def unavoidable_bytes(self) -> int:
        return 4 * self.rows * self.cols * 2 + 4 * self.cols


@dataclass(frozen=True)
class B2bWorkload:
    name: str
    op: str                # "softmax" | "gelu_tanh" | "layernorm"
    M: int
    K: int
    N1: int
    N2: int
    seed: int
    x_std: float
    w1_std: float
    w2_std: float
    b1_std: float | None = None
    alpha: float = 1.0
    description: str = ""
    kind: str = "b2b"

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.K * self.N1 + 2.0 * self.M * self.N1 * self.N2

    @property
    def unavoidable_bytes(self) -> int:
        """X, W1, b1 (gamma1, beta1), W2 read once and O written once; S never leaves the chip."""
        b = 2 * self.M * self.K + 2 * self.K * self.N1 + 2 * self.N1 * self.N2 + 2 * self.M * self.N2
        if self.b1_std is not None:
            b += 4 * self.N1
        if self.op == "layernorm":
            b += 8 * self.N1
        return b


def _c(n):
    return 1.0 / math.sqrt(n)


WORKLOADS = {
    "ln_tiny_128x512x256": GemmWorkload(
        "ln_tiny_128x512x256", "rownorm", 128, 512, 256, 0, _c(256), _c(256),
        0.1, 0.1, 0.1, "none", 1e-5,
        description="GEMM+bias+LayerNorm, tiny: X[128,256] W[256,512]"),
    "softmax_4096x2048x128": GemmWorkload(
        "softmax_4096x2048x128", "softmax", 4096, 2048, 128, 1, 1.0, _c(128),
        scale=_c(128),
        description="GEMM+row softmax: X[4096,128] W[128,2048], scale 1/sqrt(128)"),
    "gelu_ln_16384x4096x4096": GemmWorkload(
        "gelu_ln_16384x4096x4096", "rownorm", 16384, 4096, 4096, 2, _c(4096), _c(4096),
        0.02, 0.02, 0.02, "gelu_tanh", 1e-5,
        description="GEMM+bias+GELU(tanh)+LayerNorm, FFN-sized"),
    "wide_ln_8192x16384x2048": GemmWorkload(
        "wide_ln_8192x16384x2048", "rownorm", 8192, 16384, 2048, 4, _c(2048), _c(2048),
        0.1, 0.1, 0.1, "none", 1e-5,
        description="wide-row GEMM+bias+LayerNorm, row wider than one cluster"),
    "rms_16384x4096x4096": GemmWorkload(
        "rms_16384x4096x4096", "rmsnorm", 16384, 4096, 4096, 5, _c(4096), _c(4096),
        0.02, 0.02, None, "none", 1e-5,
        description="GEMM+bias+RMSNorm (gamma, no beta), FFN-sized"),
    "residual_ln_16384x4096x4096": GemmWorkload(
        "residual_ln_16384x4096x4096", "rownorm", 16384, 4096, 4096, 6, _c(4096), _c(4096),
        0.02, 0.02, 0.02, "none", 1e-5, resid_std=0.02,
        description="GEMM+bias+residual+LayerNorm (add & norm), FFN-sized"),
    "causal_softmax_4096x4096x128": GemmWorkload(
        "causal_softmax_4096x4096x128", "softmax_causal", 4096, 4096, 128, 7, 1.0, _c(128),
        scale=_c(128), mask_offset=0,
        description="GEMM+causally masked row softmax: attention scores Q[4096,128] K^T[128,4096]"),
    "b2b_attn_32768x128x1024x128": B2bWorkload(
        "b2b_attn_32768x128x1024x128", "softmax", 32768, 128, 1024, 128, 8, 1.0, _c(128), 1.0,
        alpha=_c(128),
        description="B2BGEMM with a row softmax between the GEMMs, attention-shaped: "
                    "Q[32768,128] K^T[128,1024] V[1024,128], scale 1/sqrt(128)"),
    "b2b_gelu_16384x1024x2048x128": B2bWorkload(
        "b2b_gelu_16384x1024x2048x128", "gelu_tanh", 16384, 1024, 2048, 128, 9, 1.0, _c(1024), _c(2048),
        b1_std=0.1,
        description="B2BGEMM with bias+GELU(tanh) between the GEMMs, MLP-shaped: "
                    "X[16384,1024] W1[1024,2048] W2[2048,128]"),
    "b2b_ln_16384x1024x2048x128": B2bWorkload(
        "b2b_ln_16384x1024x2048x128", "layernorm", 16384, 1024, 2048, 128, 14, 1.0, _c(1024), _c(2048),
        b1_std=0.1,
        description="B2BGEMM with bias+LayerNorm over N1 between the GEMMs: "
                    "X[16384,1024] W1[1024,2048] W2[2048,128], gamma1 ~ N(1,0.1), beta1 ~ N(0,0.1)"),
    "addln_750000x32": StitchNormWorkload(
        "addln_750000x32", "add_layernorm", 750000, 32, 10,
        description="stitched add + LayerNorm over rows, very many tiny rows"),
    "addln_64x30000": StitchNormWorkload(
        "addln_64x30000", "add_layernorm", 64, 30000, 11,
        description="stitched add + LayerNorm over rows, very few huge rows"),
    "bn_750000x32": StitchNormWorkload(
        "bn_750000x32", "batchnorm", 750000, 32, 12,
        description="stitched BatchNorm over 750000 rows (Global scheme: grid barrier, vertical packing)"),
    "bn_64x30000": StitchNormWorkload(
        "bn_64x30000", "batchnorm", 64, 30000, 13,
        description="stitched BatchNorm over 64 rows (Regional scheme: one block per column strip)"),
    "powsm_750000x32": StitchPowWorkload(
        "powsm_750000x32", 750000, 32, 16,
        description="stitched y=A+w[col]^2.5 -> row softmax, very many tiny rows (power computed once per column)"),
    "powsm_64x30000": StitchPowWorkload(
        "powsm_64x30000", 64, 30000, 17,
        description="stitched y=A+w[col]^2.5 -> row softmax, very few huge rows (power computed once per column)"),
    "stitch_750000x32": StitchWorkload(
        "stitch_750000x32", 750000, 32, 3,
        description="stitched y=A^3+b[row] -> row softmax, very many tiny rows"),
    "stitch_64x30000": StitchWorkload(
        "stitch_64x30000", 64, 30000, 3,
        description="stitched y=A^3+b[row] -> row softmax, very few huge rows"),
}


def _normal(rng, shape, std, mean=0.0):
    return (rng.standard_normal(size=shape) * std + mean).astype(np.float32)


def gemm_inputs(M: int, N: int, K: int, seed: int, *, x_std: float = 1.0,
                w_std: float = 1.0, bias_std: float | None = 0.1,
                gamma_std: float | None = 0.1, beta_std: float | None = 0.1,
                resid_std: float | None = None) -> dict:
    """X, W (bf16-valued float32) and the row-vector parameters (float32).

    A ``None`` std skips that draw (the key is then None).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    out["X"] = round_to_bf16(_normal(rng, (M, K), x_std))
    out["W"] = round_to_bf16(_normal(rng, (K, N), w_std))
    out["bias"] = None if bias_std is None else _normal(rng, (N,), bias_std)
    out["gamma"] = None if gamma_std is None else _normal(rng, (N,), gamma_std, 1.0)
    out["beta"] = None if beta_std is None else _normal(rng, (N,), beta_std)
    # drawn last, so the other draws of a seed do not depend on it
    out["R"] = None if resid_std is None else round_to_bf16(_normal(rng, (M, N), resid_std))
    return out


def stitch_inputs(rows: int, cols: int, seed: int = 3) -> dict:
    """A[rows, cols] ~ N(0, 2) fp32 and row_bias[rows] ~ U(-1, 1) fp32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A = _normal(rng, (rows, cols), 2.0)
    b = (rng.random(size=rows) * 2.0 - 1.0).astype(np.float32)
    return {"A": A, "row_bias": b}


def b2b_inputs(M: int, K: int, N1: int, N2: int, seed: int, *, x_std: float = 1.0, w1_std: float = 1.0,
               w2_std: float = 1.0, b1_std: float | None = None, ln: bool = False) -> dict:
    """X, W1, W2 (bf16-valued float32), b1 (float32, or None) and, for the
    LayerNorm epilogue, gamma1 ~ N(1, 0.1) and beta1 ~ N(0, 0.1) (float32)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    out["X"] = round_to_bf16(_normal(rng, (M, K), x_std))
    out["W1"] = round_to_bf16(_normal(rng, (K, N1), w1_std))
    out["W2"] = round_to_bf16(_normal(rng, (N1, N2), w2_std))
    out["b1"] = None if b1_std is None else _normal(rng, (N1,), b1_std)
    out["gamma1"] = _normal(rng, (N1,), 0.1, 1.0) if ln else None
    out["beta1"] = _normal(rng, (N1,), 0.1) if ln else None
    return out


def powadd_inputs(rows: int, cols: int, seed: int) -> dict:
    """A[rows, cols] ~ N(0, 1) fp32 and w[cols] ~ U(0.5, 2) fp32 (positive bases)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A = _normal(rng, (rows, cols), 1.0)
    w = (rng.random(size=cols) * 1.5 + 0.5).astype(np.float32)
    return {"A": A, "w": w}


def stitch_norm_inputs(rows: int, cols: int, seed: int, *, with_R: bool = True) -> dict:
    """A ~ N(0, 2) [rows, cols], R ~ N(0, 1) (if with_R), gamma ~ N(1, 0.1),
    beta ~ N(0, 0.1) [cols]; all fp32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {"A": _normal(rng, (rows, cols), 2.0)}
    out["R"] = _normal(rng, (rows, cols), 1.0) if with_R else None
    out["gamma"] = _normal(rng, (cols,), 0.1, 1.0)
    out["beta"] = _normal(rng, (cols,), 0.1)
    return out


def workload_inputs(name: str) -> dict:
    w = WORKLOADS[name]
    if isinstance(w, StitchWorkload):
        return stitch_inputs(w.rows, w.cols, w.seed)
    if isinstance(w, StitchNormWorkload):
        return stitch_norm_inputs(w.rows, w.cols, w.seed, with_R=w.kind == "add_layernorm")
    if isinstance(w, StitchPowWorkload):
        return powadd_inputs(w.rows, w.cols, w.seed)
    if isinstance(w, B2bWorkload):
        return b2b_inputs(w.M, w.K, w.N1, w.N2, w.seed, x_std=w.x_std, w1_std=w.w1_std, w2_std=w.w2_std,
                          b1_std=w.b1_std, ln=w.op == "layernorm")
    if w.kind in ("rownorm", "rmsnorm"):
        return gemm_inputs(w.M, w.N, w.K, w.seed, x_std=w.x_std, w_std=w.w_std,
                           bias_std=w.bias_std, gamma_std=w.gamma_std,
                           beta_std=w.beta_std, resid_std=w.resid_std)
    return gemm_inputs(w.M, w.N, w.K, w.seed, x_std=w.x_std, w_std=w.w_std,
                       bias_std=None, gamma_std=None, beta_std=None)
