// stitch.cu -- GEMM-free stitched reduce -> broadcast subgraph
//     y = A*A*A + b[row];  m = rowmax y;  s = rowsum exp(y - m);  out = exp(y - m)/s
// on irregular shapes ([AStitch] "Adaptive thread mapping": 750000x32 rows are
// packed many to a block, 64x30000 rows are split over several blocks; the
// mapping is chosen from the actual shape).
//
// Every element is read from HBM once with a 128-bit streaming load (the
// value is single-use: [sass2mlir] "Load widening and cache policy"), kept in
// registers through the whole subgraph (the exp is computed once and reused
// for the output), and written once.
//
// Two producer nodes feed the row softmax:
//   kCube:   y = a^3 + b[row]      (the pages' 750000x32 / 64x30000 subgraph)
//   kPowCol: y = a + w[col]^p      (an expensive element-wise power feeding a
//            broadcast: [AStitch] "Four stitching schemes", Regional -- every
//            CTA computes the powers of the columns it touches exactly once,
//            into shared memory, before its row loop, and every row it handles
//            reads them there: one power per column and CTA instead of one per
//            element, as register-only fusion would recompute it.  Where a CTA
//            handles a single row the producer and its consumers are one to
//            one (kPowColLocal: the power is computed with the element's load,
//            the Local scheme), as the pages' locality check would decide.)  The reduction is the three-level
// scheme of [ComFuse] (three-level reduction, Fig. 4): warp butterfly, then
// shared memory across warps, then -- when a row is split over the CTAs of a
// thread-block cluster -- distributed shared memory, peer all-to-all for few
// CTAs or leader-follower for many.
#include <cuda_runtime.h>

#include <cstdint>

#include "cf_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace cf {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = kPackedUnroll;  // row slots per thread per iteration

__device__ __forceinline__ float cube_plus(float a, float b) { return a * a * a + b; }

// kPowCol: the column powers in a shared-memory table, once per CTA (Regional:
// the CTA's rows share them); kPowColLocal: computed with each element's load
// (Local: a CTA of one row uses each power once, so a table would only add a
// phase -- the split mapping with one row per cluster)
enum StitchProd : int { kCube = 0, kPowCol = 1, kPowColLocal = 2 };

// w^p for w > 0 as 2^(p log2 w) on the MUFU (lg2.approx, ex2.approx: relative
// error about 2^-21 for |p log2 w| < 4, far inside the softmax tolerance)
__device__ __forceinline__ float pow_pos(float w, float p) { return ptx::ex2_approx(p * ptx::lg2_approx(w)); }

// the Regional producer: powers of columns [c_begin, c_end) into pw[0 ..),
// each computed by exactly one thread of the CTA, visible to all after the
// barrier.  A thread's loads of w are issued in batches of kB before any power
// is computed, so a CTA's 7500 columns cost two memory latencies, not thirty.
template <int kB>
__device__ __forceinline__ void powers_to_smem(float *pw, const float *w, float p, int c_begin, int c_end) {
    const int nt = int(blockDim.x);
    for (int c0 = c_begin + int(threadIdx.x); c0 < c_end; c0 += kB * nt) {
        float wv[kB];
#pragma unroll
        for (int k = 0; k < kB; ++k) wv[k] = (c0 + k * nt < c_end) ? __ldg(w + c0 + k * nt) : 1.f;
#pragma unroll
        for (int k = 0; k < kB; ++k)
            if (c0 + k * nt < c_end) pw[c0 + k * nt - c_begin] = pow_pos(wv[k], p);
    }
    __syncthreads();
}

// --------------------------------------------------------------------------
// Packed mapping: LPR lanes per row (horizontal packing), each lane one
// 4-column group, 32/LPR rows per warp and kUnroll row slots per thread.
// --------------------------------------------------------------------------
template <int LPR, bool VEC, int PROD>
__global__ void __launch_bounds__(kThreads) stitch_packed_kernel(const float *__restrict__ A,
                                                                 const float *__restrict__ bias,
                                                                 float *__restrict__ out, int64_t rows,
                                                                 int cols, const float *__restrict__ w, float pexp) {
    __shared__ __align__(16) float pw[PROD == kPowCol ? 4 * 32 : 1];  // the columns' powers (cols <= 128)
    constexpr int RPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (LPR - 1);
    const int rsub = lane / LPR;
    const int c0 = sub * 4;
    const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
    constexpr int64_t kRowsPerIter = int64_t(RPW) * kUnroll;
    // programmatic dependent launch: nothing in global memory before the
    // previous grid on the stream has completed
    ptx::griddep_wait();
    // kPowCol: this lane's four column powers, computed once per CTA in shared
    // memory and read once into registers for every row of the loop
    float pc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (PROD == kPowCol) {
        powers_to_smem<1>(pw, w, pexp, 0, cols);  // cols <= 128: one power per thread
#pragma unroll
        for (int j = 0; j < 4; ++j) pc[j] = (c0 + j < cols) ? pw[c0 + j] : 0.f;
    }

    bool colok[4];  // this lane's four columns exist
#pragma unroll
    for (int j = 0; j < 4; ++j) colok[j] = c0 + j < cols;
    for (int64_t base = warp * kRowsPerIter; base < rows; base += nwarps * kRowsPerIter) {
        float v[kUnroll][4];
        float bb[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t r = base + u * RPW + rsub;
            const bool rv = r < rows;
            if constexpr (VEC) {
                float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                if (rv && c0 < cols) t = __ldcs(reinterpret_cast<const float4 *>(A + r * cols + c0));
                v[u][0] = t.x;
                v[u][1] = t.y;
                v[u][2] = t.z;
                v[u][3] = t.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[u][j] = (rv && c0 + j < cols) ? __ldcs(A + r * cols + c0 + j) : 0.f;
            }
            if constexpr (PROD == kCube) bb[u] = rv ? __ldg(bias + r) : 0.f;
            else bb[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t r = base + u * RPW + rsub;
            // producer node on packed pairs; a column past the row end becomes
            // -inf (the max ignores it, its exponential is 0)
            if constexpr (PROD == kCube) {
                float s0, s1, s2, s3;
                ptx::mul2(s0, s1, v[u][0], v[u][1], v[u][0], v[u][1]);
                ptx::mul2(s2, s3, v[u][2], v[u][3], v[u][2], v[u][3]);
                ptx::fma2(v[u][0], v[u][1], s0, s1, v[u][0], v[u][1], bb[u], bb[u]);
                ptx::fma2(v[u][2], v[u][3], s2, s3, v[u][2], v[u][3], bb[u], bb[u]);
            } else {
                ptx::add2(v[u][0], v[u][1], v[u][0], v[u][1], pc[0], pc[1]);
                ptx::add2(v[u][2], v[u][3], v[u][2], v[u][3], pc[2], pc[3]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) v[u][j] = colok[j] ? v[u][j] : neg_inf();
            // every row has its column 0 in lane group position 0: m is finite
            const float m = warp_max<LPR>(fmaxf(ptx::max3(v[u][0], v[u][1], v[u][2]), v[u][3]));
            const float mL = m * kLog2e;
            float sa, sb;
            {
                float d0, d1, d2, d3;
                ptx::fma2(d0, d1, v[u][0], v[u][1], kLog2e, kLog2e, -mL, -mL);
                ptx::fma2(d2, d3, v[u][2], v[u][3], kLog2e, kLog2e, -mL, -mL);
                v[u][0] = ptx::ex2_approx(d0);
                v[u][1] = ptx::ex2_approx(d1);
                v[u][2] = ptx::ex2_approx(d2);
                v[u][3] = ptx::ex2_approx(d3);
                ptx::add2(sa, sb, v[u][0], v[u][1], v[u][2], v[u][3]);
            }
            const float inv = __frcp_rn(warp_sum<LPR>(sa + sb));
            if (r < rows) {
                if constexpr (VEC) {
                    if (c0 < cols) {
                        float4 y;
                        ptx::mul2(y.x, y.y, v[u][0], v[u][1], inv, inv);
                        ptx::mul2(y.z, y.w, v[u][2], v[u][3], inv, inv);
                        __stcs(reinterpret_cast<float4 *>(out + r * cols + c0), y);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (colok[j]) __stcs(out + r * cols + c0 + j, v[u][j] * inv);
                }
            }
        }
    }
    // the next grid may be scheduled once this CTA's rows are written
    ptx::griddep_launch_dependents();
}

// --------------------------------------------------------------------------
// Split mapping: one row per cluster of C CTAs (task splitting).  CTA `rank`
// owns 4-column groups [rank*gpc, rank*gpc + gpc); each thread holds up to V
// groups in registers.
// --------------------------------------------------------------------------
template <int V, bool VEC, int PROD>
__global__ void __launch_bounds__(kThreads) stitch_split_kernel(const float *__restrict__ A,
                                                                const float *__restrict__ bias,
                                                                float *__restrict__ out, int64_t rows, int cols,
                                                                int gpc, int leader, uint32_t *err,
                                                                unsigned long long tmo, const float *__restrict__ w,
                                                                float pexp) {
    extern __shared__ __align__(16) float pws[];  // kPowCol: powers of this CTA's 4 gpc columns
    __shared__ MaxSum red[kThreads / 32];
    __shared__ __align__(16) MaxSum slot[2][16];  // level-3 partials, by row parity
    __shared__ __align__(16) MaxSum res[2];       // leader's result, by row parity
    __shared__ __align__(8) uint64_t xbar[2];     // exchange barriers, by row parity
    __shared__ uint32_t abort_flag;

    const uint32_t C = ptx::cluster_nctarank();
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t cid = ptx::cluster_id_x();
    const uint32_t ncl = ptx::nclusters_x();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int ng = (cols + 3) >> 2;
    const int g0 = int(rank) * gpc;
    const int g1 = min(ng, g0 + gpc);
    volatile uint32_t *abort = &abort_flag;

    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&xbar[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&xbar[1]), 1);
        abort_flag = 0u;
        ptx::fence_mbarrier_init_cluster();
    }
    __syncthreads();
    // Peers may signal these barriers once every CTA of the cluster initialised
    // its own: arrive now, wait just before the first exchange (the first row's
    // loads are in flight in between).
    ptx::cluster_arrive_relaxed();
    // programmatic dependent launch: nothing in global memory before the
    // previous grid on the stream has completed
    ptx::griddep_wait();
    int it = 0;
    for (int64_t row = cid; row < rows; row += ncl, ++it) {
        const int par = it & 1;
        const uint32_t xb = ptx::smem_u32(&xbar[par]);
        const uint32_t xph = uint32_t(it >> 1) & 1u;
        const float *a = A + row * cols;
        float *o = out + row * cols;
        const float bb = PROD == kCube ? __ldg(bias + row) : 0.f;

        float e[V][4];
        float wl[PROD == kPowColLocal ? V : 1][4];  // kPowColLocal: the columns' bases, loaded with A
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int g = g0 + threadIdx.x + v * kThreads;
            if constexpr (VEC) {
                float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                if (g < g1) t = __ldcs(reinterpret_cast<const float4 *>(a) + g);
                e[v][0] = t.x;
                e[v][1] = t.y;
                e[v][2] = t.z;
                e[v][3] = t.w;
                if constexpr (PROD == kPowColLocal) {
                    float4 b4 = make_float4(1.f, 1.f, 1.f, 1.f);
                    if (g < g1) b4 = __ldg(reinterpret_cast<const float4 *>(w) + g);
                    wl[v][0] = b4.x;
                    wl[v][1] = b4.y;
                    wl[v][2] = b4.z;
                    wl[v][3] = b4.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    e[v][j] = (g < g1 && 4 * g + j < cols) ? __ldcs(a + 4 * g + j) : 0.f;
                    if constexpr (PROD == kPowColLocal) wl[v][j] = (g < g1 && 4 * g + j < cols) ? __ldg(w + 4 * g + j) : 1.f;
                }
            }
        }
        // kPowCol: the powers of this CTA's columns, once, into shared memory (the
        // cluster's rows all reuse them), computed while the first row's loads fly
        if (PROD == kPowCol && it == 0) powers_to_smem<16>(pws, w, pexp, 4 * g0, min(cols, 4 * g1));
        if (it == 0) ptx::cluster_wait_acquire();
        // producer node; a column outside the row slice becomes -inf, so the max
        // ignores it and its exponential is 0 without further tests
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int g = g0 + threadIdx.x + v * kThreads;
            if constexpr (PROD == kCube) {  // a^3 + b on packed pairs
                float s0, s1, s2, s3;
                ptx::mul2(s0, s1, e[v][0], e[v][1], e[v][0], e[v][1]);
                ptx::mul2(s2, s3, e[v][2], e[v][3], e[v][2], e[v][3]);
                ptx::fma2(e[v][0], e[v][1], s0, s1, e[v][0], e[v][1], bb, bb);
                ptx::fma2(e[v][2], e[v][3], s2, s3, e[v][2], e[v][3], bb, bb);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = VEC ? g < g1 : (g < g1 && 4 * g + j < cols);
                if constexpr (PROD == kPowColLocal) e[v][j] += pow_pos(wl[v][j], pexp);
                else if constexpr (PROD == kPowCol) e[v][j] += ok ? pws[4 * (g - g0) + j] : 0.f;
                e[v][j] = ok ? e[v][j] : neg_inf();
            }
        }
        // thread-local aggregation: max (three-input), then the sum of the
        // exponentials on packed pairs (kept for the output)
        float mt = neg_inf();
#pragma unroll
        for (int v = 0; v < V; ++v) mt = ptx::max3(ptx::max3(mt, e[v][0], e[v][1]), e[v][2], e[v][3]);
        const float mL = mt == neg_inf() ? 0.f : mt * kLog2e;  // no column: every exponent is -inf
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) {
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                float d0, d1;
                ptx::fma2(d0, d1, e[v][j], e[v][j + 1], kLog2e, kLog2e, -mL, -mL);
                e[v][j] = ptx::ex2_approx(d0);  // 2^-inf = 0
                e[v][j + 1] = ptx::ex2_approx(d1);
                ptx::add2(sa, sb, sa, sb, e[v][j], e[v][j + 1]);
            }
        }
        const float st = sa + sb;
        // level 1 (warp): the max in one redux, each lane's sum rescaled to it,
        // then a butterfly of plain sums (no exponential on the shuffle chain)
        const float mw = ptx::warp_redux_max(mt);
        const float sw = warp_sum<32>(mt == neg_inf() ? 0.f : st * ptx::ex2_approx((mt - mw) * kLog2e));
        // level 2: across the CTA's warps through shared memory, the same way (a
        // full-warp sum, so every lane that sends below holds the CTA's total)
        if (lane == 0) red[warp] = MaxSum{mw, sw};
        __syncthreads();
        if (warp == 0) {
            const MaxSum q = (lane < kThreads / 32) ? red[lane] : MaxSum{neg_inf(), 0.f};
            const float mc = ptx::warp_redux_max(q.m);
            const float sc = warp_sum<32>(q.m == neg_inf() ? 0.f : q.s * ptx::ex2_approx((q.m - mc) * kLog2e));
            if (!*abort) {
                // level 3: an 8-byte st.async of this CTA's (max, sum) into the
                // gathering CTAs' shared memory, completing on their barrier; lane r
                // sends to CTA r, so the remote stores are in flight together
                const uint32_t my_slot = ptx::smem_u32(&slot[par][rank]);
                if (!leader) {
                    if (lane == 0) ptx::mbar_arrive_expect_tx(xb, C * 8u);
                    if (uint32_t(lane) < C)
                        ptx::st_async_f2(ptx::mapa(my_slot, uint32_t(lane)), mc, sc, ptx::mapa(xb, uint32_t(lane)));
                } else if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(xb, rank == 0 ? C * 8u : 8u);
                    ptx::st_async_f2(ptx::mapa(my_slot, 0), mc, sc, ptx::mapa(xb, 0));
                }
            }
        }
        // the row's statistics from the C partials, max first and then the
        // rescaled sums, in rank order (every CTA folds them identically)
        MaxSum tot;
        if (!leader || rank == 0) {
            ptx::mbar_wait_bounded<true>(xb, xph, tmo, abort, err, 0x70000000u | uint32_t(par));
            float m = slot[par][0].m;
            for (uint32_t r = 1; r < C; ++r) m = fmaxf(m, slot[par][r].m);
            float sum = 0.f;
            for (uint32_t r = 0; r < C; ++r)
                sum += slot[par][r].m == neg_inf() ? 0.f : slot[par][r].s * ptx::ex2_approx((slot[par][r].m - m) * kLog2e);
            tot = MaxSum{m, sum};
            if (leader && warp == 0 && !*abort && lane >= 1 && uint32_t(lane) < C) {
                // the leader sends the row statistics back to the followers (lane r to CTA r)
                const uint32_t res_addr = ptx::smem_u32(&res[par]);
                ptx::st_async_f2(ptx::mapa(res_addr, uint32_t(lane)), tot.m, tot.s, ptx::mapa(xb, uint32_t(lane)));
            }
        } else {
            ptx::mbar_wait_bounded<true>(xb, xph, tmo, abort, err, 0x70000010u | uint32_t(par));
            tot = res[par];
        }
        // broadcast back over the row: out = exp(y - mt) * exp(mt - m) / s
        const float f = (mt == neg_inf()) ? 0.f : ptx::ex2_approx((mt - tot.m) * kLog2e) / tot.s;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int g = g0 + threadIdx.x + v * kThreads;
            if constexpr (VEC) {
                if (g < g1) {
                    float4 y;
                    ptx::mul2(y.x, y.y, e[v][0], e[v][1], f, f);
                    ptx::mul2(y.z, y.w, e[v][2], e[v][3], f, f);
                    __stcs(reinterpret_cast<float4 *>(o) + g, y);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (g < g1 && 4 * g + j < cols) __stcs(o + 4 * g + j, e[v][j] * f);
            }
        }
        // slot[par] / res[par] are written again two rows later: a peer sends for
        // row it+2 only after this CTA sent for row it+1, which its thread 0 does
        // after the barrier above that every thread passes once done with row it
    }
    // the next grid may be scheduled once this CTA's rows are written
    ptx::griddep_launch_dependents();
    // No CTA leaves while a peer may still access its shared memory (every
    // incoming st.async was waited for; this covers the outgoing ones).
    ptx::cluster_arrive_relaxed();
    ptx::cluster_wait_acquire();
}

template <int LPR, bool VEC>
void *packed_fn(int prod) {
    return prod == kPowCol ? reinterpret_cast<void *>(&stitch_packed_kernel<LPR, VEC, kPowCol>)
                           : reinterpret_cast<void *>(&stitch_packed_kernel<LPR, VEC, kCube>);
}

void *packed_kernel(int lpr, bool vec, int prod = kCube) {
    switch (lpr) {
        case 1: return vec ? packed_fn<1, true>(prod) : packed_fn<1, false>(prod);
        case 2: return vec ? packed_fn<2, true>(prod) : packed_fn<2, false>(prod);
        case 4: return vec ? packed_fn<4, true>(prod) : packed_fn<4, false>(prod);
        case 8: return vec ? packed_fn<8, true>(prod) : packed_fn<8, false>(prod);
        case 16: return vec ? packed_fn<16, true>(prod) : packed_fn<16, false>(prod);
        case 32: return vec ? packed_fn<32, true>(prod) : packed_fn<32, false>(prod);
        default: return nullptr;
    }
}

template <int V, bool VEC>
void *split_fn(int prod) {
    if (prod == kPowCol) return reinterpret_cast<void *>(&stitch_split_kernel<V, VEC, kPowCol>);
    if (prod == kPowColLocal) return reinterpret_cast<void *>(&stitch_split_kernel<V, VEC, kPowColLocal>);
    return reinterpret_cast<void *>(&stitch_split_kernel<V, VEC, kCube>);
}

void *split_kernel(int v, bool vec, int prod) {
    switch (v) {
        case 1: return vec ? split_fn<1, true>(prod) : split_fn<1, false>(prod);
        case 2: return vec ? split_fn<2, true>(prod) : split_fn<2, false>(prod);
        case 4: return vec ? split_fn<4, true>(prod) : split_fn<4, false>(prod);
        case 8: return vec ? split_fn<8, true>(prod) : split_fn<8, false>(prod);
        case 16: return vec ? split_fn<16, true>(prod) : split_fn<16, false>(prod);
        default: return nullptr;
    }
}

}  // namespace

int stitch_packed_blocks_per_sm(int lpr, bool vec) {
    // cached per (device, variant): no occupancy query under stream capture
    static int cache[64][6][2] = {};
    void *fn = packed_kernel(lpr, vec);
    if (!fn) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int li = 0;
    while ((1 << li) < lpr) ++li;
    int &c = cache[dev][li][vec ? 1 : 0];
    if (c == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        c = n;
    }
    return c;
}

cudaError_t launch_stitch(const StitchPlan &p, const float *A, const float *bias, float *out, int64_t rows,
                          int64_t cols, uint32_t *err, cudaStream_t stream, const float *w, float pexp) {
    const int prod = w != nullptr ? kPowCol : kCube;
    if (p.mapping == 1) {
        void *fn = packed_kernel(p.lpr, p.vec, prod);
        if (!fn) return cudaErrorInvalidValue;
        int icols = int(cols);
        void *args[] = {(void *)&A, (void *)&bias, (void *)&out, (void *)&rows, (void *)&icols, (void *)&w,
                        (void *)&pexp};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(p.grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = p.pdl ? 1 : 0;
        return cudaLaunchKernelExC(&cfg, fn, args);
    }
    if (p.mapping == 2) {
        // one row per cluster: each power is used once per CTA (Local scheme);
        // several: the CTA's rows share a shared-memory table (Regional)
        const int sprod = (prod == kPowCol && int64_t(p.grid / p.cluster) >= rows) ? int(kPowColLocal) : prod;
        void *fn = split_kernel(p.per_thread, p.vec, sprod);
        if (!fn) return cudaErrorInvalidValue;
        const int ng = int((cols + 3) / 4);
        int gpc = (ng + p.cluster - 1) / p.cluster;
        // kPowCol: the CTA's column powers in dynamic shared memory
        const int smem = sprod == kPowCol ? gpc * 16 : 0;
        {
            // attributes once per (device, variant): non-portable clusters, and the
            // largest power table seen
            static bool done[64][5][2][3] = {};
            static int set_smem[64][5][2] = {};
            int dev = 0;
            cudaError_t e = cudaGetDevice(&dev);
            if (e != cudaSuccess) return e;
            int vi = 0;
            while ((1 << vi) < p.per_thread) ++vi;
            if (dev < 0 || dev >= 64 || vi > 4) return cudaErrorInvalidValue;
            if (p.cluster > 8 && !done[dev][vi][p.vec ? 1 : 0][sprod]) {
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
                done[dev][vi][p.vec ? 1 : 0][sprod] = true;
            }
            if (smem > 48 * 1024 && smem > set_smem[dev][vi][p.vec ? 1 : 0]) {
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                if (e != cudaSuccess) return e;
                set_smem[dev][vi][p.vec ? 1 : 0] = smem;
            }
        }
        int icols = int(cols);
        int leader = p.leader;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(p.grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
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
        unsigned long long tmo = p.timeout_ns;
        void *args[] = {(void *)&A, (void *)&bias, (void *)&out, (void *)&rows, (void *)&icols, (void *)&gpc,
                        (void *)&leader, (void *)&err, (void *)&tmo, (void *)&w, (void *)&pexp};
        return cudaLaunchKernelExC(&cfg, fn, args);
    }
    return cudaErrorInvalidValue;
}

}  // namespace cf
