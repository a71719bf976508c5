// stitch_norm.cu -- GEMM-free stitched normalisation subgraphs, each one
// kernel ([AStitch] "Four stitching schemes", "Adaptive thread mapping"):
//
//  * add + LayerNorm over rows:  x = A + R;  out = (x - mean)/sqrt(var + eps)
//    * gamma[col] + beta[col].  An elementwise producer (Local), two row
//    reductions (mean, then the variance around it, two passes over values
//    held in registers) and their broadcast; the column parameters are a
//    one-to-many dependency, loaded once per thread and reused for every row
//    it handles.  Thread mapping as for the stitched softmax: rows of up to
//    128 columns packed several to a warp, wider rows split over the CTAs of a
//    cluster with one DSMEM exchange of (mean, M2) per row.
//
//  * BatchNorm over columns (batch statistics):  out = (A - mean_col) /
//    sqrt(var_col + eps) * gamma[col] + beta[col].  The statistic of a column
//    depends on every row.
//      - Regional (few rows): one CTA holds all rows of a 128-column strip in
//        registers; warps combine their column partials in shared memory and
//        normalise from registers.  One HBM pass.
//      - Global (many rows): vertical packing -- one resident wave of CTAs,
//        each owning a contiguous row range of a column strip; column
//        partials go to global memory, an in-kernel grid barrier replaces
//        the kernel boundary, every CTA folds all partials in one fixed order
//        (so all hold bitwise-equal statistics) and normalises its rows,
//        re-reading them from L2 (first read under an evict-last policy).
//    The choice is the pages' block-locality check: a column's producers and
//    consumers fit one block (Regional) or they do not (Global).
//
// Every wait is bounded by %globaltimer; a timeout records
// CF_ERR_DEVICE_TIMEOUT in the workspace error word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/cf.h"
#include "cf_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace cf {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = kPackedUnroll;  // row slots per thread per iteration (packed rows)
constexpr int kGlobalThreads = 512;  // Global BatchNorm: ~100 registers a thread, no spills
constexpr int kGlobalUnroll = 8;     // its row slots per thread in flight (4 KB per warp)

// float4 group g of a row; zeros past `cols` (scalar path) or past `g1`
template <bool VEC>
__device__ __forceinline__ float4 load_group(const float *row, int g, int cols, bool ok) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!ok) return t;
    if constexpr (VEC) {
        t = __ldcs(reinterpret_cast<const float4 *>(row) + g);
    } else {
        const int c = 4 * g;
        t.x = __ldcs(row + c);
        if (c + 1 < cols) t.y = __ldcs(row + c + 1);
        if (c + 2 < cols) t.z = __ldcs(row + c + 2);
        if (c + 3 < cols) t.w = __ldcs(row + c + 3);
    }
    return t;
}

template <bool VEC>
__device__ __forceinline__ void store_group(float *row, int g, int cols, float4 v) {
    if constexpr (VEC) {
        __stcs(reinterpret_cast<float4 *>(row) + g, v);
    } else {
        const int c = 4 * g;
        __stcs(row + c, v.x);
        if (c + 1 < cols) __stcs(row + c + 1, v.y);
        if (c + 2 < cols) __stcs(row + c + 2, v.z);
        if (c + 3 < cols) __stcs(row + c + 3, v.w);
    }
}

template <bool VEC>
__device__ __forceinline__ float4 ldg_group(const float *p, int g, int cols) {
    if constexpr (VEC) return __ldg(reinterpret_cast<const float4 *>(p) + g);
    float4 t;
    const int c = 4 * g;
    t.x = __ldg(p + c);
    t.y = c + 1 < cols ? __ldg(p + c + 1) : 0.f;
    t.z = c + 2 < cols ? __ldg(p + c + 2) : 0.f;
    t.w = c + 3 < cols ? __ldg(p + c + 3) : 0.f;
    return t;
}

// 16-byte asynchronous global -> shared copy (L2 only, no L1 allocation);
// complete for this thread after cp_async_wait_all
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }

// valid lanes of a 4-group starting at column c
__device__ __forceinline__ float nvalid4(int c, int cols) { return float(max(0, min(4, cols - c))); }

// ==========================================================================
// add + LayerNorm, packed rows (LPR lanes per row, one 4-column group each)
// ==========================================================================
template <int LPR, bool VEC>
__global__ void __launch_bounds__(kThreads) addln_packed_kernel(const float *__restrict__ A,
                                                                const float *__restrict__ R,
                                                                const float *__restrict__ gamma,
                                                                const float *__restrict__ beta,
                                                                float *__restrict__ out, int64_t rows, int cols,
                                                                float eps) {
    constexpr int RPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int g = lane & (LPR - 1);
    const int rsub = lane / LPR;
    const int c0 = 4 * g;
    const bool gv = c0 < cols;
    const float inv_n = 1.0f / float(cols);
    const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
    constexpr int64_t kRowsPerIter = int64_t(RPW) * kUnroll;
    ptx::griddep_wait();
    // column parameters: loaded once, reused for every row this thread handles
    const float4 ga = gv ? ldg_group<VEC>(gamma, g, cols) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 be = gv ? ldg_group<VEC>(beta, g, cols) : make_float4(0.f, 0.f, 0.f, 0.f);

    for (int64_t base = warp * kRowsPerIter; base < rows; base += nwarps * kRowsPerIter) {
        float4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t r = base + u * RPW + rsub;
            const bool ok = r < rows && gv;
            x[u] = load_group<VEC>(A + r * cols, g, cols, ok);
            if (R != nullptr) x[u] = add4(x[u], load_group<VEC>(R + r * cols, g, cols, ok));
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t r = base + u * RPW + rsub;
            // two passes over the row held in registers: mean, then M2 about it
            float s = (x[u].x + x[u].y) + (x[u].z + x[u].w);  // invalid lanes hold 0
            s = warp_sum<LPR>(s);
            const float mean = s * inv_n;
            float4 d = make_float4(x[u].x - mean, x[u].y - mean, x[u].z - mean, x[u].w - mean);
            if (!gv) d = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!VEC) {
                if (c0 + 1 >= cols) d.y = 0.f;
                if (c0 + 2 >= cols) d.z = 0.f;
                if (c0 + 3 >= cols) d.w = 0.f;
            }
            float q = fmaf(d.x, d.x, fmaf(d.y, d.y, fmaf(d.z, d.z, d.w * d.w)));
            q = warp_sum<LPR>(q);
            const float rstd = rsqrtf(fmaf(q, inv_n, eps));
            if (r < rows && gv) {
                const float4 y = make_float4(fmaf(d.x * rstd, ga.x, be.x), fmaf(d.y * rstd, ga.y, be.y),
                                             fmaf(d.z * rstd, ga.z, be.z), fmaf(d.w * rstd, ga.w, be.w));
                store_group<VEC>(out + r * cols, g, cols, y);
            }
        }
    }
    ptx::griddep_launch_dependents();
}

// ==========================================================================
// add + LayerNorm, one row per cluster of C CTAs (task splitting).  CTA
// `rank` owns 4-column groups [rank*gpc, rank*gpc + gpc); each thread holds
// up to V groups.  One DSMEM exchange of the CTA's (mean, M2) per row.
// ==========================================================================
template <int V, bool VEC>
__global__ void __launch_bounds__(kThreads) addln_split_kernel(const float *__restrict__ A,
                                                               const float *__restrict__ R,
                                                               const float *__restrict__ gamma,
                                                               const float *__restrict__ beta,
                                                               float *__restrict__ out, int64_t rows, int cols,
                                                               float eps, int gpc, uint32_t *err,
                                                               unsigned long long tmo) {
    __shared__ float reds[kThreads / 32];         // the warps' sums
    __shared__ float redq[kThreads / 32];         // the warps' squared deviations
    __shared__ __align__(16) MeanM2 slot[2][16];  // per-CTA partials, by row parity
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ uint32_t abort_flag;
    // 128-bit rows, up to 4 groups a thread: this thread's gamma and beta
    // groups copied into shared memory under the first row's loads (no
    // registers held across the reduction; every row reuses them)
    constexpr bool kGB = VEC && V <= 4;
    __shared__ __align__(16) float4 gbs[kGB ? 2 * V * kThreads : 1];

    const uint32_t C = ptx::cluster_nctarank();
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t cid = ptx::cluster_id_x();
    const uint32_t ncl = ptx::nclusters_x();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int ng = (cols + 3) >> 2;
    const int g0 = int(rank) * gpc;
    const int g1 = min(ng, g0 + gpc);
    // columns of CTA r's slice (the same for every row)
    auto slice_count = [&](int r) {
        const int ga = r * gpc, gb = min(ng, ga + gpc);
        return gb > ga ? float(min(cols, 4 * gb) - 4 * ga) : 0.f;
    };
    const float ncta = slice_count(int(rank));
    volatile uint32_t *abort = &abort_flag;

    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&xbar[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&xbar[1]), 1);
        abort_flag = 0u;
        ptx::fence_mbarrier_init_cluster();
    }
    __syncthreads();
    ptx::cluster_arrive_relaxed();
    ptx::griddep_wait();

    int it = 0;
    for (int64_t row = cid; row < rows; row += ncl, ++it) {
        const int par = it & 1;
        const uint32_t xb = ptx::smem_u32(&xbar[par]);
        const uint32_t xph = uint32_t(it >> 1) & 1u;
        const float *a = A + row * cols;
        const float *rr = R != nullptr ? R + row * cols : nullptr;
        float4 x[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int g = g0 + threadIdx.x + v * kThreads;
            const bool ok = g < g1;
            x[v] = load_group<VEC>(a, g, cols, ok);
            if (rr != nullptr) x[v] = add4(x[v], load_group<VEC>(rr, g, cols, ok));
        }
        if (it == 0) {
            // gamma and beta of this CTA's columns (the same for every row) into
            // shared memory, or into L1, under the first row's loads, so the
            // output pass after the exchange does not wait on L2 for them
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int g = g0 + threadIdx.x + v * kThreads;
                if (g < g1) {
                    if constexpr (kGB) {
                        cp_async_16(ptx::smem_u32(&gbs[v * kThreads + threadIdx.x]), gamma + 4 * g);
                        cp_async_16(ptx::smem_u32(&gbs[(V + v) * kThreads + threadIdx.x]), beta + 4 * g);
                    } else {
                        ptx::prefetch_l1(gamma + 4 * g);
                        ptx::prefetch_l1(beta + 4 * g);
                    }
                }
            }
            if constexpr (kGB) cp_async_commit();
            ptx::cluster_wait_acquire();
        }
        // the CTA's mean (levels 1 and 2 on plain sums: missing columns hold 0)
        float st = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) st += (x[v].x + x[v].y) + (x[v].z + x[v].w);
        st = warp_sum<32>(st);
        if (lane == 0) reds[warp] = st;
        __syncthreads();
        float scta = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) scta += reds[w];
        const float mc = ncta > 0.f ? scta / ncta : 0.f;
        // the squared deviations from it, over this thread's existing columns
        float qa = 0.f, qb = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int g = g0 + threadIdx.x + v * kThreads;
            if (g < g1) {
                float d0, d1, d2, d3;
                ptx::add2(d0, d1, x[v].x, x[v].y, -mc, -mc);
                ptx::add2(d2, d3, x[v].z, x[v].w, -mc, -mc);
                if constexpr (!VEC) {  // a row's last group may be partial
                    const int c = 4 * g;
                    d1 = c + 1 < cols ? d1 : 0.f;
                    d2 = c + 2 < cols ? d2 : 0.f;
                    d3 = c + 3 < cols ? d3 : 0.f;
                }
                ptx::fma2(qa, qb, d0, d1, d0, d1, qa, qb);
                ptx::fma2(qa, qb, d2, d3, d2, d3, qa, qb);
            }
        }
        const float qt = warp_sum<32>(qa + qb);
        if (lane == 0) redq[warp] = qt;
        __syncthreads();
        if (warp == 0) {
            const float qc = warp_sum<32>(lane < kThreads / 32 ? redq[lane] : 0.f);
            if (!*abort) {
                // level 3: this CTA's (mean, M2) into every CTA's slot, lane r to CTA r
                const uint32_t my_slot = ptx::smem_u32(&slot[par][rank]);
                if (lane == 0) ptx::mbar_arrive_expect_tx(xb, C * 8u);
                if (uint32_t(lane) < C)
                    ptx::st_async_f2(ptx::mapa(my_slot, uint32_t(lane)), mc, qc, ptx::mapa(xb, uint32_t(lane)));
            }
        }
        ptx::mbar_wait_bounded<true>(xb, xph, tmo, abort, err, 0x71000000u | uint32_t(par));
        // the row's statistics from the C partials (counts known from the
        // slices), in rank order: mean = sum(n_r mean_r) / N, then
        // M2 = sum(M2_r + n_r (mean_r - mean)^2)
        float sm = 0.f;
        for (uint32_t r = 0; r < C; ++r) sm = fmaf(slice_count(int(r)), slot[par][r].mean, sm);
        const float mean = sm / float(cols);
        float m2 = 0.f;
        for (uint32_t r = 0; r < C; ++r) {
            const float d = slot[par][r].mean - mean;
            m2 += fmaf(slice_count(int(r)) * d, d, slot[par][r].m2);
        }
        const float rstd = rsqrtf(fmaf(m2, 1.0f / float(cols), eps));
        float *o = out + row * cols;
        if constexpr (kGB) {
            if (it == 0) cp_async_wait_all();  // this thread's own copies
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int g = g0 + threadIdx.x + v * kThreads;
            if (g < g1) {
                float4 ga, be;
                if constexpr (kGB) {
                    ga = gbs[v * kThreads + threadIdx.x];
                    be = gbs[(V + v) * kThreads + threadIdx.x];
                } else {
                    ga = ldg_group<VEC>(gamma, g, cols);
                    be = ldg_group<VEC>(beta, g, cols);
                }
                const float4 y = make_float4(fmaf((x[v].x - mean) * rstd, ga.x, be.x),
                                             fmaf((x[v].y - mean) * rstd, ga.y, be.y),
                                             fmaf((x[v].z - mean) * rstd, ga.z, be.z),
                                             fmaf((x[v].w - mean) * rstd, ga.w, be.w));
                store_group<VEC>(o, g, cols, y);
            }
        }
        // slot[par] is written again two rows later: a peer sends for row it+2
        // only after this CTA sent for row it+1, which its warp 0 does after
        // the barriers above that every thread passes once done with row it
    }
    ptx::griddep_launch_dependents();
    ptx::cluster_arrive_relaxed();
    ptx::cluster_wait_acquire();
}

// ==========================================================================
// BatchNorm, Regional: one CTA per 128-column strip holds all rows (warp w
// takes rows w, w+8, ...; RPT of them) in registers.
// ==========================================================================
template <int RPT, bool VEC>
__global__ void __launch_bounds__(kThreads) bn_regional_kernel(const float *__restrict__ A,
                                                               const float *__restrict__ gamma,
                                                               const float *__restrict__ beta,
                                                               float *__restrict__ out, float *__restrict__ mean_out,
                                                               float *__restrict__ var_out, int rows, int cols,
                                                               float eps) {
    __shared__ float2 red[kThreads / 32][128];
    __shared__ float4 stat[32][3];  // per 4-group: mean, gamma*rstd, beta
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ng = (cols + 3) >> 2;
    const int g = blockIdx.x * 32 + lane;
    const bool gv = g < ng;
    ptx::griddep_wait();
    // gamma and beta of the column this thread folds below, loaded with the rows
    // (an L2 round trip after the fold otherwise)
    const int tcol = blockIdx.x * 128 + int(threadIdx.x);
    const bool tc = threadIdx.x < 128 && tcol < cols;
    const float gcol = tc ? __ldg(gamma + tcol) : 0.f;
    const float bcol = tc ? __ldg(beta + tcol) : 0.f;
    float4 x[RPT];
    float n = 0.f;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int r = warp + 8 * k;
        const bool ok = gv && r < rows;
        x[k] = load_group<VEC>(A + int64_t(r) * cols, g, cols, ok);
        if (r < rows) n += 1.f;
        s = add4(s, x[k]);
    }
    const float in = n > 0.f ? 1.0f / n : 0.f;
    const float4 m = make_float4(s.x * in, s.y * in, s.z * in, s.w * in);
    float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        if (warp + 8 * k < rows) {
            const float dx = x[k].x - m.x, dy = x[k].y - m.y, dz = x[k].z - m.z, dw = x[k].w - m.w;
            q.x = fmaf(dx, dx, q.x);
            q.y = fmaf(dy, dy, q.y);
            q.z = fmaf(dz, dz, q.z);
            q.w = fmaf(dw, dw, q.w);
        }
    }
    red[warp][4 * lane + 0] = make_float2(m.x, q.x);
    red[warp][4 * lane + 1] = make_float2(m.y, q.y);
    red[warp][4 * lane + 2] = make_float2(m.z, q.z);
    red[warp][4 * lane + 3] = make_float2(m.w, q.w);
    __syncthreads();
    if (threadIdx.x < 128) {
        // fold the 8 warps' partials of column t in warp order (warp w holds rows
        // w, w + 8, ...): mean = sum(n_w mean_w) / rows, then
        // M2 = sum(M2_w + n_w (mean_w - mean)^2)
        const int t = threadIdx.x;
        const int col = tcol;
        float sm = 0.f;
#pragma unroll 1
        for (int w = 0; w < kThreads / 32; ++w) sm = fmaf(float(rows > w ? (rows - w + 7) / 8 : 0), red[w][t].x, sm);
        const float mean = sm / float(rows);
        float m2 = 0.f;
#pragma unroll 1
        for (int w = 0; w < kThreads / 32; ++w) {
            const float d = red[w][t].x - mean;
            m2 += fmaf(float(rows > w ? (rows - w + 7) / 8 : 0) * d, d, red[w][t].y);
        }
        const MeanM2 acc{mean, m2};
        const float var = acc.m2 / float(rows);
        const float sc = rsqrtf(var + eps);
        float *st = reinterpret_cast<float *>(&stat[0][0]);
        if (col < cols) {
            st[(t >> 2) * 12 + 0 + (t & 3)] = acc.mean;
            st[(t >> 2) * 12 + 4 + (t & 3)] = gcol * sc;
            st[(t >> 2) * 12 + 8 + (t & 3)] = bcol;
            if (mean_out != nullptr) mean_out[col] = acc.mean;
            if (var_out != nullptr) var_out[col] = var;
        }
    }
    __syncthreads();
    if (gv) {
        const float4 mu = stat[lane][0], sc = stat[lane][1], be = stat[lane][2];
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
            const int r = warp + 8 * k;
            if (r < rows) {
                const float4 y = make_float4(fmaf(x[k].x - mu.x, sc.x, be.x), fmaf(x[k].y - mu.y, sc.y, be.y),
                                             fmaf(x[k].z - mu.z, sc.z, be.z), fmaf(x[k].w - mu.w, sc.w, be.w));
                store_group<VEC>(out + int64_t(r) * cols, g, cols, y);
            }
        }
    }
    ptx::griddep_launch_dependents();
}

// ==========================================================================
// BatchNorm, Global: grid = strips x chunks CTAs, all resident (vertical
// packing).  CTA b works on strip b % strips (LPR 4-column groups) and the
// rows of chunk b / strips.
// ==========================================================================
template <int LPR, bool VEC>
__global__ void __launch_bounds__(kGlobalThreads, 1) bn_global_kernel(
    const float *__restrict__ A, const float *__restrict__ gamma, const float *__restrict__ beta,
    float *__restrict__ out, float *__restrict__ mean_out, float *__restrict__ var_out, int64_t rows, int cols,
    float eps, int strips, uint32_t *err, uint32_t *counters, float2 *partials, int extra_arrivals,
    unsigned long long tmo) {
    constexpr int RPW = 32 / LPR;          // row slots per warp
    constexpr int kWarps = kGlobalThreads / 32;
    constexpr int W = 4 * LPR;             // columns of a strip
    __shared__ float2 red[kWarps][W];
    __shared__ float redn[kWarps];
    __shared__ float4 stat[LPR][3];        // per 4-group: mean, gamma*rstd, beta
    __shared__ uint32_t abort_flag;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ng = (cols + 3) >> 2;
    const int strip = int(blockIdx.x) % strips;
    const int chunk = int(blockIdx.x) / strips;
    const int nchunks = int(gridDim.x) / strips;
    const int sub = lane & (LPR - 1), rsub = lane / LPR;
    const int g = strip * LPR + sub;
    const bool gv = g < ng;
    const int64_t r0 = rows * chunk / nchunks, r1 = rows * (chunk + 1) / nchunks;
    const int slot = warp * RPW + rsub;
    constexpr int S = kWarps * RPW;        // row slots of the CTA
    volatile uint32_t *abort = &abort_flag;
    if (threadIdx.x == 0) abort_flag = 0u;
    ptx::griddep_wait();
    const uint64_t keep = ptx::policy_evict_last();

    // ---- pass 1: running (n, mean, M2) per column over this CTA's rows, in
    // chunks of kGlobalUnroll rows (two passes over each chunk held in registers)
    float n = 0.f;
    MeanM2 run[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    for (int64_t base = r0 + slot; base < r1; base += int64_t(S) * kGlobalUnroll) {
        float4 x[kGlobalUnroll];
        float nc = 0.f;
#pragma unroll
        for (int u = 0; u < kGlobalUnroll; ++u) {
            const int64_t r = base + int64_t(u) * S;
            const bool ok = r < r1;
            x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ok && gv) {
                const float *row = A + r * cols;
                if constexpr (VEC) {
                    x[u] = ptx::ld_f4_hint(reinterpret_cast<const float4 *>(row) + g, keep);
                } else {
                    const int c = 4 * g;
                    x[u].x = ptx::ld_f32_hint(row + c, keep);
                    if (c + 1 < cols) x[u].y = ptx::ld_f32_hint(row + c + 1, keep);
                    if (c + 2 < cols) x[u].z = ptx::ld_f32_hint(row + c + 2, keep);
                    if (c + 3 < cols) x[u].w = ptx::ld_f32_hint(row + c + 3, keep);
                }
            }
            if (ok) nc += 1.f;
        }
        if (nc == 0.f) break;
        const float ic = 1.0f / nc;
        float mc[4] = {0.f, 0.f, 0.f, 0.f}, qc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < kGlobalUnroll; ++u) {
            mc[0] += x[u].x;
            mc[1] += x[u].y;
            mc[2] += x[u].z;
            mc[3] += x[u].w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) mc[j] *= ic;
#pragma unroll
        for (int u = 0; u < kGlobalUnroll; ++u) {
            if (base + int64_t(u) * S < r1) {
                const float d[4] = {x[u].x - mc[0], x[u].y - mc[1], x[u].z - mc[2], x[u].w - mc[3]};
#pragma unroll
                for (int j = 0; j < 4; ++j) qc[j] = fmaf(d[j], d[j], qc[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) run[j] = combine_counts_safe(run[j], n, MeanM2{mc[j], qc[j]}, nc);
        n += nc;
    }
    // ---- CTA reduce: row slots of a warp (lanes LPR apart), then the warps
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float nj = n;
        warp_meanm2<RPW, LPR>(run[j], nj);
        if (j == 3) n = nj;
    }
    if (rsub == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) red[warp][4 * sub + j] = make_float2(run[j].mean, run[j].m2);
        if (sub == 0) redn[warp] = n;
    }
    __syncthreads();
    if (threadIdx.x < W) {
        const int t = threadIdx.x;
        MeanM2 acc{red[0][t].x, red[0][t].y};
        float na = redn[0];
        for (int w = 1; w < kWarps; ++w) {
            acc = combine_counts_safe(acc, na, MeanM2{red[w][t].x, red[w][t].y}, redn[w]);
            na += redn[w];
        }
        // this CTA's partial of column strip*W + t (its count follows from r0, r1)
        partials[size_t(blockIdx.x) * W + t] = make_float2(acc.mean, acc.m2);
        __threadfence();
    }
    __syncthreads();
    // ---- grid barrier: every CTA of the launch is resident (host-checked)
    if (threadIdx.x == 0) {
        const uint32_t want = gridDim.x + uint32_t(extra_arrivals);
        ptx::red_add_release_gpu(counters, 1u);
        const uint64_t t0 = ptx::globaltimer();
        uint32_t spins = 0;
        while (ptx::ld_acquire_gpu(counters) < want) {
            if ((++spins & 63u) == 0u) {
                if (ptx::globaltimer() - t0 > tmo) {
                    *abort = 1u;
                    ptx::record_error(err, 7u /*CF_ERR_DEVICE_TIMEOUT*/, 0x72000000u | blockIdx.x);
                    break;
                }
                if (ptx::ld_relaxed_gpu(err) != 0u) {  // another CTA gave up: do not wait out the bound
                    *abort = 1u;
                    break;
                }
            }
        }
    }
    __syncthreads();
    if (*abort) {
        ptx::griddep_launch_dependents();
        return;
    }
    // ---- fold every chunk's partial of the strip's columns, one warp per
    // column, lanes over chunks, in one fixed order (bitwise-equal in all CTAs)
    for (int t = warp; t < W; t += kWarps) {
        MeanM2 acc{0.f, 0.f};
        float na = 0.f;
        for (int c = lane; c < nchunks; c += 32) {
            const float2 pc = ptx::ld_relaxed_gpu_f2(partials + size_t(c * strips + strip) * W + t);
            const float nc = float(rows * (c + 1) / nchunks - rows * c / nchunks);
            acc = combine_counts_safe(acc, na, MeanM2{pc.x, pc.y}, nc);
            na += nc;
        }
        warp_meanm2<32>(acc, na);
        if (lane == 0) {
            const int col = strip * W + t;
            const float var = na > 0.f ? acc.m2 / na : 0.f;
            float *st = reinterpret_cast<float *>(&stat[0][0]);
            if (col < cols) {
                st[(t >> 2) * 12 + 0 + (t & 3)] = acc.mean;
                st[(t >> 2) * 12 + 4 + (t & 3)] = __ldg(gamma + col) * rsqrtf(var + eps);
                st[(t >> 2) * 12 + 8 + (t & 3)] = __ldg(beta + col);
                if (chunk == 0) {
                    if (mean_out != nullptr) mean_out[col] = acc.mean;
                    if (var_out != nullptr) var_out[col] = var;
                }
            } else {
                st[(t >> 2) * 12 + 0 + (t & 3)] = 0.f;
                st[(t >> 2) * 12 + 4 + (t & 3)] = 0.f;
                st[(t >> 2) * 12 + 8 + (t & 3)] = 0.f;
            }
        }
    }
    __syncthreads();
    // ---- departure: the last CTA to leave the barrier resets the counters
    if (threadIdx.x == 0) {
        const uint32_t d = ptx::atom_add_relaxed_gpu(counters + 1, 1u);
        if (d == gridDim.x - 1u) {
            ptx::st_relaxed_gpu(counters, 0u);
            ptx::st_relaxed_gpu(counters + 1, 0u);
        }
    }
    // ---- pass 2: normalise the same rows (an L2 hit for rows kept evict-last)
    const float4 mu = gv ? stat[sub][0] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 sc = gv ? stat[sub][1] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 be = gv ? stat[sub][2] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (gv) {
        for (int64_t base = r0 + slot; base < r1; base += int64_t(S) * kGlobalUnroll) {
            float4 x[kGlobalUnroll];
#pragma unroll
            for (int u = 0; u < kGlobalUnroll; ++u) {
                const int64_t r = base + int64_t(u) * S;
                x[u] = load_group<VEC>(A + r * cols, g, cols, r < r1);
            }
#pragma unroll
            for (int u = 0; u < kGlobalUnroll; ++u) {
                const int64_t r = base + int64_t(u) * S;
                if (r < r1) {
                    const float4 y = make_float4(fmaf(x[u].x - mu.x, sc.x, be.x), fmaf(x[u].y - mu.y, sc.y, be.y),
                                                 fmaf(x[u].z - mu.z, sc.z, be.z), fmaf(x[u].w - mu.w, sc.w, be.w));
                    store_group<VEC>(out + r * cols, g, cols, y);
                }
            }
        }
    }
    ptx::griddep_launch_dependents();
}

// ==========================================================================
// BatchNorm, Global, streamed through shared memory by TMA.  A CTA's rows (a
// contiguous range of one column strip, aligned to the stage height) are read
// twice: once for the statistics and once, after the grid barrier, to be
// normalised and stored (from registers, streaming stores).  The CTA's shared
// memory holds kTmaBufBytes of stage buffers: `ring` of them stream (the
// first pass loads those stages evict-last, so that the second pass finds
// them in L2), the others keep the CTA's first `res` stages resident from the
// first pass to the second.  Those are the oldest loads of the first pass,
// the ones the L2 is likeliest to have dropped by the time the second pass
// (with the output's writes) comes to them; they are loaded evict-first and
// normalised first.  The producer issues the second pass's ring loads while
// the grid barrier is in progress.  One producer warp, eight compute warps; a
// compute thread owns one 4-column group of the strip and RPS rows of every
// stage.
// ==========================================================================
constexpr int kTmaBufBytes = 13 * 16384;  // stage buffers per CTA (ring + resident)
constexpr int kTmaMaxRing = 32;
constexpr int kTmaMaxRes = 48;
constexpr int kTmaCompute = 256;
constexpr int kTmaThreads = kTmaCompute + 32;

template <int LPR>
struct BnTmaShape {
    static constexpr int W = 4 * LPR;                                  // strip columns
    static constexpr int BR = (1024 / LPR) < 256 ? (1024 / LPR) : 256;  // stage rows (box height <= 256)
    static constexpr int STAGE = W * BR * 4;                           // bytes (4, 8 or 16 KB)
    static constexpr int SLOTS = kTmaCompute / LPR;                    // row slots
    static constexpr int RPS = BR / SLOTS;                             // rows per thread per stage
};

// kFlat: the strip is the whole row (cols == 4*LPR), so a stage is one
// contiguous block of memory and moves by one untiled bulk copy each way
template <int LPR, bool kFlat>
__global__ void __launch_bounds__(kTmaThreads, 1) bn_global_tma_kernel(const __grid_constant__ BnTmaArgs a) {
    using Sh = BnTmaShape<LPR>;
    constexpr int W = Sh::W, BR = Sh::BR, STAGE = Sh::STAGE, SLOTS = Sh::SLOTS, RPS = Sh::RPS;
    constexpr int kCW = kTmaCompute / 32;
    extern __shared__ __align__(128) uint8_t ring_smem[];
    __shared__ float2 red[kCW][W];
    __shared__ float redn[kCW];
    __shared__ float4 stat[LPR][3];  // per 4-group: mean, gamma*rstd, beta
    __shared__ __align__(8) uint64_t full[kTmaMaxRing];
    __shared__ __align__(8) uint64_t empty[kTmaMaxRing];
    __shared__ __align__(8) uint64_t fullr[kTmaMaxRes];  // resident stages: one load each
    __shared__ uint32_t abort_flag;

    const uint32_t bufs = ptx::smem_u32(ring_smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int strip = int(blockIdx.x) % a.strips;
    const int chunk = int(blockIdx.x) / a.strips;
    const int nchunks = int(gridDim.x) / a.strips;
    const int ring = a.ring;  // host-clamped: 2 <= ring <= kTmaMaxRing, ring + res buffers fit
    const int64_t r0 = int64_t(chunk) * a.rows_per_chunk;
    const int64_t r1 = r0 + a.rows_per_chunk < a.rows ? r0 + a.rows_per_chunk : a.rows;
    const int nst = r1 > r0 ? int((r1 - r0 + BR - 1) / BR) : 0;  // stages per pass
    const int nres = a.res < nst ? a.res : nst;                   // resident stages (the first ones)
    const int nstream = nst - nres;                               // ring stages per pass
    volatile uint32_t *abort = &abort_flag;
    const uint64_t tmo = a.timeout_ns;
    unsigned long long *const tr = a.trace != nullptr ? a.trace + size_t(blockIdx.x) * CF_TRACE_SLOTS : nullptr;
    if (threadIdx.x == 0) {
        if (tr != nullptr) tr[0] = ptx::globaltimer();
        for (int s = 0; s < ring; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty[s]), kCW);
        }
        for (int j = 0; j < nres; ++j) ptx::mbar_init(ptx::smem_u32(&fullr[j]), 1);
        abort_flag = 0u;
        ptx::fence_mbarrier_init_cluster();
    }
    __syncthreads();
    ptx::griddep_wait();

    if (warp == kCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tensormap(&a.tmap_a);
            const uint64_t keep = ptx::policy_evict_last(), once = ptx::policy_evict_first();
            // stage `st` of this CTA's rows into buffer `dst`, completing on `bar`
            auto load = [&](int st, uint32_t dst, uint32_t bar, uint64_t pol) {
                const int64_t row = r0 + int64_t(st) * BR;
                if constexpr (kFlat) {
                    // the rows of this stage that exist (a multiple of 16 bytes: cols % 4 == 0)
                    const int64_t nrow = r1 - row < BR ? r1 - row : BR;
                    const uint32_t bytes = uint32_t(nrow) * uint32_t(W) * 4u;
                    ptx::mbar_arrive_expect_tx(bar, bytes);
                    ptx::bulk_load_g2s_hint(dst, a.A + row * W, bytes, bar, pol);
                } else {
                    ptx::mbar_arrive_expect_tx(bar, uint32_t(STAGE));
                    ptx::tma_load_2d_hint(dst, &a.tmap_a, bar, strip * W, int(row), pol);
                }
            };
            for (int j = 0; j < nres; ++j) load(j, bufs + (ring + j) * STAGE, ptx::smem_u32(&fullr[j]), once);
            uint32_t s = 0, ph = 0;
            int issued = 0;
            for (int i = 0; i < 2 * nstream; ++i) {
                if (!ptx::mbar_wait_bounded(ptx::smem_u32(&empty[s]), ph ^ 1u, tmo, abort, a.err, 0x73000000u | s))
                    break;
                load(nres + (i < nstream ? i : i - nstream), bufs + s * STAGE, ptx::smem_u32(&full[s]),
                     i < nstream ? keep : once);
                ++issued;
                if (++s == uint32_t(ring)) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // every issued load has landed before the CTA may exit
            volatile uint32_t local_abort = 0;
            for (int j = 0; j < nres; ++j)
                ptx::mbar_wait_bounded(ptx::smem_u32(&fullr[j]), 0u, tmo, &local_abort, nullptr, 0);
            for (int i = issued > ring ? issued - ring : 0; i < issued; ++i)
                ptx::mbar_wait_bounded(ptx::smem_u32(&full[i % ring]), uint32_t(i / ring) & 1u, tmo, &local_abort,
                                       nullptr, 0);
        }
        return;
    }

    // ---------------------------------------------------------------- compute
    const int c = threadIdx.x;
    const int sub = c % LPR, slot = c / LPR;
    uint32_t s = 0, ph = 0;
    // ---- pass 1: running (n, mean, M2) of this thread's 4 columns
    float n = 0.f;
    MeanM2 run[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    for (int i = 0; i < nst; ++i) {
        const bool res = i < nres;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(res ? &fullr[i] : &full[s]), res ? 0u : ph, tmo, abort, a.err,
                                    0x74000000u | (res ? 0x100u + uint32_t(i) : s)))
            break;
        const float4 *st4 = reinterpret_cast<const float4 *>(ring_smem + (res ? ring + i : int(s)) * STAGE);
        const int64_t rb = r0 + int64_t(i) * BR;
        float4 x[RPS];
        float nc = 0.f;
#pragma unroll
        for (int k = 0; k < RPS; ++k) {
            const int lr = slot + k * SLOTS;
            x[k] = st4[lr * LPR + sub];
            if (rb + lr < r1) nc += 1.f;
            else x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!res) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));
            if (++s == uint32_t(ring)) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (nc == 0.f) continue;
        const float ic = 1.0f / nc;
        float mc[4] = {0.f, 0.f, 0.f, 0.f}, qc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < RPS; ++k) {
            mc[0] += x[k].x;
            mc[1] += x[k].y;
            mc[2] += x[k].z;
            mc[3] += x[k].w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) mc[j] *= ic;
#pragma unroll
        for (int k = 0; k < RPS; ++k) {
            if (rb + slot + k * SLOTS < r1) {
                const float d[4] = {x[k].x - mc[0], x[k].y - mc[1], x[k].z - mc[2], x[k].w - mc[3]};
#pragma unroll
                for (int j = 0; j < 4; ++j) qc[j] = fmaf(d[j], d[j], qc[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) run[j] = combine_counts_safe(run[j], n, MeanM2{mc[j], qc[j]}, nc);
        n += nc;
    }
    // ---- CTA reduce: lanes LPR apart hold the same columns, then the warps
    constexpr int RPW = 32 / LPR;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float nj = n;
        warp_meanm2<RPW, LPR>(run[j], nj);
        if (j == 3) n = nj;
    }
    if (lane < LPR) {
#pragma unroll
        for (int j = 0; j < 4; ++j) red[warp][4 * sub + j] = make_float2(run[j].mean, run[j].m2);
        if (lane == 0) redn[warp] = n;
    }
    ptx::named_bar_sync(1, kTmaCompute);
    if (c < W) {
        MeanM2 acc{red[0][c].x, red[0][c].y};
        float na = redn[0];
        for (int w = 1; w < kCW; ++w) {
            acc = combine_counts_safe(acc, na, MeanM2{red[w][c].x, red[w][c].y}, redn[w]);
            na += redn[w];
        }
        a.partials[size_t(blockIdx.x) * W + c] = make_float2(acc.mean, acc.m2);
        __threadfence();
    }
    ptx::named_bar_sync(1, kTmaCompute);
    // ---- grid barrier (every CTA resident: host-checked)
    if (c == 0) {
        if (tr != nullptr) tr[1] = ptx::globaltimer();
        const uint32_t want = gridDim.x + uint32_t(a.extra_arrivals);
        ptx::red_add_release_gpu(a.counters, 1u);
        const uint64_t t0 = ptx::globaltimer();
        uint32_t spins = 0;
        while (ptx::ld_acquire_gpu(a.counters) < want) {
            if ((++spins & 63u) == 0u) {
                if (ptx::globaltimer() - t0 > tmo) {
                    *abort = 1u;
                    ptx::record_error(a.err, 7u /*CF_ERR_DEVICE_TIMEOUT*/, 0x72000000u | blockIdx.x);
                    break;
                }
                if (ptx::ld_relaxed_gpu(a.err) != 0u) {
                    *abort = 1u;
                    break;
                }
            }
        }
    }
    ptx::named_bar_sync(1, kTmaCompute);
    if (*abort) return;
    if (c == 0 && tr != nullptr) tr[2] = ptx::globaltimer();
    // ---- fold every chunk's partial of the strip: one warp per column, lanes
    // over chunks, one fixed order (bitwise-equal statistics in all CTAs)
    for (int t = warp; t < W; t += kCW) {
        MeanM2 acc{0.f, 0.f};
        float na = 0.f;
        for (int k = lane; k < nchunks; k += 32) {
            const float2 pc = ptx::ld_relaxed_gpu_f2(a.partials + size_t(k * a.strips + strip) * W + t);
            const int64_t q0 = int64_t(k) * a.rows_per_chunk;
            const int64_t q1 = q0 + a.rows_per_chunk < a.rows ? q0 + a.rows_per_chunk : a.rows;
            const float nk = q1 > q0 ? float(q1 - q0) : 0.f;
            acc = combine_counts_safe(acc, na, MeanM2{pc.x, pc.y}, nk);
            na += nk;
        }
        warp_meanm2<32>(acc, na);
        if (lane == 0) {
            const int col = strip * W + t;
            float *st = reinterpret_cast<float *>(&stat[0][0]);
            const float var = na > 0.f ? acc.m2 / na : 0.f;
            const bool cv = col < a.cols;
            st[(t >> 2) * 12 + 0 + (t & 3)] = cv ? acc.mean : 0.f;
            st[(t >> 2) * 12 + 4 + (t & 3)] = cv ? __ldg(a.gamma + col) * rsqrtf(var + a.eps) : 0.f;
            st[(t >> 2) * 12 + 8 + (t & 3)] = cv ? __ldg(a.beta + col) : 0.f;
            if (cv && chunk == 0) {
                if (a.mean_out != nullptr) a.mean_out[col] = acc.mean;
                if (a.var_out != nullptr) a.var_out[col] = var;
            }
        }
    }
    ptx::named_bar_sync(1, kTmaCompute);
    if (c == 0) {  // departure: the last CTA to leave the barrier resets the counters
        const uint32_t d = ptx::atom_add_relaxed_gpu(a.counters + 1, 1u);
        if (d == gridDim.x - 1u) {
            ptx::st_relaxed_gpu(a.counters, 0u);
            ptx::st_relaxed_gpu(a.counters + 1, 0u);
        }
    }
    // ---- pass 2: normalise each stage and store it from registers (the
    // resident stages first: they are already in shared memory).  A ring
    // stage goes back to the producer as soon as its rows are in registers,
    // as in the first pass, so no store holds a stage.
    const float4 mu = stat[sub][0], sc = stat[sub][1], be = stat[sub][2];
    const bool gv = kFlat || (strip * LPR + sub) * 4 < a.cols;  // this thread's column group exists
    float *const ocol = a.out + (kFlat ? 0 : strip * W) + 4 * sub;
    const int ostride = kFlat ? W : a.cols;
    for (int i = 0; i < nst; ++i) {
        const bool res = i < nres;
        if (!res && !ptx::mbar_wait_bounded(ptx::smem_u32(&full[s]), ph, tmo, abort, a.err, 0x75000000u | s)) break;
        const float4 *st4 = reinterpret_cast<const float4 *>(ring_smem + (res ? ring + i : int(s)) * STAGE);
        float4 x[RPS];
#pragma unroll
        for (int k = 0; k < RPS; ++k) x[k] = st4[(slot + k * SLOTS) * LPR + sub];
        if (!res) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&empty[s]));
            if (++s == uint32_t(ring)) {
                s = 0;
                ph ^= 1u;
            }
        }
        const int64_t rb = r0 + int64_t(i) * BR;
#pragma unroll
        for (int k = 0; k < RPS; ++k) {
            const int64_t row = rb + slot + k * SLOTS;
            if (gv && row < r1)
                __stcs(reinterpret_cast<float4 *>(ocol + row * ostride),
                       make_float4(fmaf(x[k].x - mu.x, sc.x, be.x), fmaf(x[k].y - mu.y, sc.y, be.y),
                                   fmaf(x[k].z - mu.z, sc.z, be.z), fmaf(x[k].w - mu.w, sc.w, be.w)));
        }
    }
    if (c == 0 && tr != nullptr) tr[3] = ptx::globaltimer();
    ptx::griddep_launch_dependents();
}

// --------------------------------------------------------------------------
// kernel tables
// --------------------------------------------------------------------------
template <int LPR>
void *addln_packed_fn(bool vec) {
    return vec ? reinterpret_cast<void *>(&addln_packed_kernel<LPR, true>)
               : reinterpret_cast<void *>(&addln_packed_kernel<LPR, false>);
}
void *addln_packed_kernel_for(int lpr, bool vec) {
    switch (lpr) {
        case 1: return addln_packed_fn<1>(vec);
        case 2: return addln_packed_fn<2>(vec);
        case 4: return addln_packed_fn<4>(vec);
        case 8: return addln_packed_fn<8>(vec);
        case 16: return addln_packed_fn<16>(vec);
        case 32: return addln_packed_fn<32>(vec);
        default: return nullptr;
    }
}
template <int V>
void *addln_split_fn(bool vec) {
    return vec ? reinterpret_cast<void *>(&addln_split_kernel<V, true>)
               : reinterpret_cast<void *>(&addln_split_kernel<V, false>);
}
void *addln_split_kernel_for(int v, bool vec) {
    switch (v) {
        case 1: return addln_split_fn<1>(vec);
        case 2: return addln_split_fn<2>(vec);
        case 4: return addln_split_fn<4>(vec);
        case 8: return addln_split_fn<8>(vec);
        case 16: return addln_split_fn<16>(vec);
        default: return nullptr;
    }
}
template <int RPT>
void *bn_regional_fn(bool vec) {
    return vec ? reinterpret_cast<void *>(&bn_regional_kernel<RPT, true>)
               : reinterpret_cast<void *>(&bn_regional_kernel<RPT, false>);
}
void *bn_regional_kernel_for(int rpt, bool vec) {
    switch (rpt) {
        case 1: return bn_regional_fn<1>(vec);
        case 2: return bn_regional_fn<2>(vec);
        case 4: return bn_regional_fn<4>(vec);
        case 8: return bn_regional_fn<8>(vec);
        case 16: return bn_regional_fn<16>(vec);
        case 32: return bn_regional_fn<32>(vec);
        default: return nullptr;
    }
}
template <int LPR>
void *bn_global_fn(bool vec) {
    return vec ? reinterpret_cast<void *>(&bn_global_kernel<LPR, true>)
               : reinterpret_cast<void *>(&bn_global_kernel<LPR, false>);
}
void *bn_global_kernel_for(int lpr, bool vec) {
    switch (lpr) {
        case 1: return bn_global_fn<1>(vec);
        case 2: return bn_global_fn<2>(vec);
        case 4: return bn_global_fn<4>(vec);
        case 8: return bn_global_fn<8>(vec);
        case 16: return bn_global_fn<16>(vec);
        case 32: return bn_global_fn<32>(vec);
        default: return nullptr;
    }
}

cudaError_t launch_plain(void *fn, int grid, int threads, bool pdl, cudaStream_t stream, void **args) {
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

int blocks_per_sm_cached(void *fn, int threads, int key) {
    static int cache[64][64] = {};
    int dev = 0;
    if (!fn || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || key < 0 || key >= 64) return 0;
    int &c = cache[dev][key];
    if (c == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        c = n;
    }
    return c;
}

template <int LPR>
void *bn_tma_fn(bool flat) {
    return flat ? reinterpret_cast<void *>(&bn_global_tma_kernel<LPR, true>)
                : reinterpret_cast<void *>(&bn_global_tma_kernel<LPR, false>);
}
void *bn_tma_kernel_for(int lpr, bool flat) {
    switch (lpr) {
        case 1: return bn_tma_fn<1>(flat);
        case 2: return bn_tma_fn<2>(flat);
        case 4: return bn_tma_fn<4>(flat);
        case 8: return bn_tma_fn<8>(flat);
        case 16: return bn_tma_fn<16>(flat);
        case 32: return bn_tma_fn<32>(flat);
        default: return nullptr;
    }
}
int bn_tma_stage_bytes(int lpr) { return 4 * lpr * std::min(256, 1024 / lpr) * 4; }

int log2i(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

}  // namespace

int addln_packed_blocks_per_sm(int lpr, bool vec) {
    return blocks_per_sm_cached(addln_packed_kernel_for(lpr, vec), kThreads, log2i(lpr) * 2 + (vec ? 1 : 0));
}

int bn_global_blocks_per_sm(int lpr, bool vec) {
    return blocks_per_sm_cached(bn_global_kernel_for(lpr, vec), kGlobalThreads, 32 + log2i(lpr) * 2 + (vec ? 1 : 0));
}

int bn_tma_box_rows(int lpr) { return std::min(256, 1024 / lpr); }

void bn_tma_buffers(int lpr, int stages, int *ring, int *res) {
    const int nbuf = kTmaBufBytes / bn_tma_stage_bytes(lpr);
    // default: 128 KB of streaming stages per CTA (750000x32: 8 of 16 KB, 5
    // resident; 50.9 us against 51.9 with 12 streaming and none resident)
    int r = stages > 0 ? stages : (128 * 1024) / bn_tma_stage_bytes(lpr);
    r = std::max(2, std::min(r, std::min(nbuf, kTmaMaxRing)));
    *ring = r;
    *res = std::min(nbuf - r, kTmaMaxRes);
}

int bn_tma_blocks_per_sm(int lpr) {
    static int cache[64][6] = {};
    void *fn = bn_tma_kernel_for(lpr, false);
    int dev = 0;
    if (!fn || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int &c = cache[dev][log2i(lpr)];
    if (c == 0) {
        const int smem = kTmaBufBytes;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kTmaThreads, smem) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        c = n;
    }
    return c;
}

cudaError_t launch_batchnorm_tma(int lpr, const BnTmaArgs &a, int grid, bool pdl, cudaStream_t stream) {
    void *fn = bn_tma_kernel_for(lpr, a.flat != 0);
    if (!fn) return cudaErrorInvalidValue;
    const int smem = kTmaBufBytes;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void *args[] = {(void *)&a};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_add_layernorm(const StitchPlan &p, const float *A, const float *R, const float *gamma,
                                 const float *beta, float *out, int64_t rows, int64_t cols, float eps, uint32_t *err,
                                 cudaStream_t stream) {
    int icols = int(cols);
    if (p.mapping == 1) {
        void *args[] = {(void *)&A, (void *)&R, (void *)&gamma, (void *)&beta, (void *)&out, (void *)&rows,
                        (void *)&icols, (void *)&eps};
        return launch_plain(addln_packed_kernel_for(p.lpr, p.vec), p.grid, kThreads, p.pdl, stream, args);
    }
    if (p.mapping != 2) return cudaErrorInvalidValue;
    void *fn = addln_split_kernel_for(p.per_thread, p.vec);
    if (!fn) return cudaErrorInvalidValue;
    if (p.cluster > 8) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const int ng = int((cols + 3) / 4);
    int gpc = (ng + p.cluster - 1) / p.cluster;
    unsigned long long tmo = p.timeout_ns;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    void *args[] = {(void *)&A, (void *)&R, (void *)&gamma, (void *)&beta, (void *)&out, (void *)&rows,
                    (void *)&icols, (void *)&eps, (void *)&gpc, (void *)&err, (void *)&tmo};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_batchnorm(const BnPlan &p, const float *A, const float *gamma, const float *beta, float *out,
                             float *mean_out, float *var_out, int64_t rows, int64_t cols, float eps, uint32_t *err,
                             uint32_t *counters, float2 *partials, cudaStream_t stream) {
    int icols = int(cols);
    if (p.mapping == 3) {
        int irows = int(rows);
        void *args[] = {(void *)&A, (void *)&gamma, (void *)&beta, (void *)&out, (void *)&mean_out,
                        (void *)&var_out, (void *)&irows, (void *)&icols, (void *)&eps};
        return launch_plain(bn_regional_kernel_for(p.rpt, p.vec), p.grid, kThreads, p.pdl, stream, args);
    }
    if (p.mapping != 4) return cudaErrorInvalidValue;
    int strips = p.strips;
    int extra = p.extra_arrivals;
    unsigned long long tmo = p.timeout_ns;
    void *args[] = {(void *)&A, (void *)&gamma, (void *)&beta, (void *)&out, (void *)&mean_out, (void *)&var_out,
                    (void *)&rows, (void *)&icols, (void *)&eps, (void *)&strips, (void *)&err, (void *)&counters,
                    (void *)&partials, (void *)&extra, (void *)&tmo};
    return launch_plain(bn_global_kernel_for(p.lpr, p.vec), p.grid, kGlobalThreads, p.pdl, stream, args);
}

}  // namespace cf
