// rowstats.cuh -- statistics carried by the row reductions and their combine
// operators, used at every level of the three-level reduction ([ComFuse]
// three-level reduction scheme, Fig. 4): thread-local aggregation over a
// fragment, warp butterfly shuffles, warp-group combine through shared
// memory, and inter-CTA aggregation over distributed shared memory (and, for
// rows wider than a cluster, a global-memory partial buffer).
//
// Two statistics are needed by the epilogues here:
//  * LayerNorm: (mean, M2) of n values, M2 = sum (x - mean)^2, combined with
//    Chan et al.'s pairwise update; n is implicit (every partial of one level
//    covers the same number of columns).
//  * Softmax: (m, s) with m = max z, s = sum exp(z - m), combined by
//    rescaling the smaller-max side ("online softmax").
// Combines happen in a fixed order everywhere, so every CTA that combines the
// same partials obtains bitwise-identical statistics, and repeated launches
// are bitwise reproducible (no floating-point atomics).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace cf {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// The GELU node (tanh form): 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))),
// tanh by the tanh.approx.f32 instruction.
__device__ __forceinline__ float gelu_tanh_dev(float x) {
    const float k0 = 0.7978845608028654f;
    const float k1 = 0.044715f;
    const float u = k0 * fmaf(k1 * x, x * x, x);
    return 0.5f * x * (1.0f + ptx::tanh_approx(u));
}

// GELU(tanh) on a packed pair: 0.5 x (1 + tanh(x (c0 + c0 c1 x^2))), the two
// tanh on the MUFU
__device__ __forceinline__ void gelu_tanh_pair(float &x0, float &x1) {
    constexpr float c0 = 0.7978845608028654f;                 // sqrt(2 / pi)
    constexpr float c01 = 0.7978845608028654f * 0.044715f;    // sqrt(2 / pi) * 0.044715
    float q0, q1, u0, u1, h0, h1;
    ptx::mul2(q0, q1, x0, x1, x0, x1);                 // x^2
    ptx::fma2(q0, q1, q0, q1, c01, c01, c0, c0);       // c0 + c0 c1 x^2
    ptx::mul2(u0, u1, q0, q1, x0, x1);                 // the tanh argument
    ptx::mul2(h0, h1, x0, x1, 0.5f, 0.5f);             // x / 2
    const float t0 = ptx::tanh_approx(u0), t1 = ptx::tanh_approx(u1);
    ptx::fma2(x0, x1, h0, h1, t0, t1, h0, h1);         // x/2 + x/2 tanh
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// --------------------------------------------------------------------------
// LayerNorm statistics
// --------------------------------------------------------------------------
struct MeanM2 {
    float mean;
    float m2;
};

// Combine two partials over the same count n each; result covers 2n.
__device__ __forceinline__ MeanM2 combine_equal(MeanM2 a, MeanM2 b, float n) {
    const float d = b.mean - a.mean;
    MeanM2 r;
    r.mean = a.mean + 0.5f * d;
    r.m2 = a.m2 + b.m2 + d * d * (0.5f * n);
    return r;
}

// Fold partial b (count nb) into running a (count na).  The weight nb / n uses
// the fast division intrinsic (within 2 ulp for these counts): the IEEE
// division's out-of-line slow path would force the callers' register arrays
// (the fixed-order folds) into local memory.
__device__ __forceinline__ MeanM2 combine_counts(MeanM2 a, float na, MeanM2 b, float nb) {
    const float n = na + nb;
    const float d = b.mean - a.mean;
    const float f = __fdividef(nb, n);
    MeanM2 r;
    r.mean = a.mean + d * f;
    r.m2 = a.m2 + b.m2 + d * d * (na * f);
    return r;
}

// As combine_counts, for partials that may be empty (count 0 on either side).
__device__ __forceinline__ MeanM2 combine_counts_safe(MeanM2 a, float na, MeanM2 b, float nb) {
    if (nb == 0.f) return a;
    if (na == 0.f) return b;
    return combine_counts(a, na, b, nb);
}

// level-1 butterfly of (count, mean, M2) partials over groups of `width`
// lanes spaced `stride` apart (lower lane first: every lane folds the same
// pairs in the same order, so all lanes end with bitwise-equal results)
template <int kWidth, int kStride = 1>
__device__ __forceinline__ void warp_meanm2(MeanM2 &v, float &n) {
#pragma unroll
    for (int off = kStride; off < kWidth * kStride; off <<= 1) {
        MeanM2 o;
        o.mean = __shfl_xor_sync(0xffffffffu, v.mean, off);
        o.m2 = __shfl_xor_sync(0xffffffffu, v.m2, off);
        const float no = __shfl_xor_sync(0xffffffffu, n, off);
        const bool upper = (threadIdx.x & off) != 0;
        v = upper ? combine_counts_safe(o, no, v, n) : combine_counts_safe(v, n, o, no);
        n += no;
    }
}

// (mean, M2) of 32 values held by one thread: two passes over registers.
__device__ __forceinline__ MeanM2 chunk_mean_m2(const float (&x)[32]) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) s += x[j];
    const float mean = s * (1.0f / 32.0f);
    float m2 = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float d = x[j] - mean;
        m2 = fmaf(d, d, m2);
    }
    return MeanM2{mean, m2};
}

// --------------------------------------------------------------------------
// Softmax statistics
// --------------------------------------------------------------------------
struct MaxSum {
    float m;
    float s;
};

__device__ __forceinline__ MaxSum combine_maxsum(MaxSum a, MaxSum b) {
    const float m = fmaxf(a.m, b.m);
    MaxSum r;
    r.m = m;
    if (m == neg_inf()) {
        r.s = 0.f;
    } else {
        r.s = a.s * ptx::ex2_approx((a.m - m) * kLog2e) + b.s * ptx::ex2_approx((b.m - m) * kLog2e);
    }
    return r;
}

// --------------------------------------------------------------------------
// level 1: warp butterfly over groups of `width` lanes (power of two)
// --------------------------------------------------------------------------
template <int kWidth>
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = kWidth / 2; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

template <int kWidth>
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = kWidth / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <int kWidth>
__device__ __forceinline__ MaxSum warp_maxsum(MaxSum v) {
#pragma unroll
    for (int off = kWidth / 2; off > 0; off >>= 1) {
        MaxSum o;
        o.m = __shfl_xor_sync(0xffffffffu, v.m, off);
        o.s = __shfl_xor_sync(0xffffffffu, v.s, off);
        // lower lane first: every lane folds the same pair in the same order
        v = (threadIdx.x & off) ? combine_maxsum(o, v) : combine_maxsum(v, o);
    }
    return v;
}

}  // namespace cf
