// gemm_fused.cu -- one persistent sm_103a kernel computing a bf16 GEMM and,
// in the same kernel, a dependency-rich epilogue whose row reductions span
// many tiles and CTAs:
//     LN:       y = LayerNorm(alpha*acc + bias) * gamma + beta
//     GELU_LN:  y = LayerNorm(GELU_tanh(alpha*acc + bias)) * gamma + beta
//               (with GemmArgs::rms, RMSNorm in place of LayerNorm for both; with
//               GemmArgs::resid, a bf16 residual added after the activation)
//     SOFTMAX:  y = softmax(scale*acc + bias)   (SOFTMAX_MASK: over the causally
//               masked row, keeping column j of row i iff j <= i + offset)
//
// Design (GB300-first; the page mechanisms it realises are cited inline):
//  * Tiles are 128 rows x n_slice columns (n_slice <= 256; or 512, a wide
//    tile filling all of tensor memory, which both epilogue groups share, one
//    half of its columns each).  A row block's
//    N / n_slice tiles go to the CTAs of one thread-block cluster (CTA rank
//    r -> column slice r), so all CTAs of one reduction are co-scheduled
//    ([ComFuse] Stage-Stream Execution Model, cluster mapping).  Rows wider
//    than one cluster are split over G clusters that meet through a
//    global-memory partial buffer and an in-kernel counter barrier
//    ([AStitch] "Global" stitching scheme; [sass2mlir] "Grid-barrier
//    synthesis").
//  * Warp roles: warp 0 issues TMA loads of X and W tiles into an S-stage
//    shared-memory ring; warp 1 allocates tensor memory and issues
//    tcgen05.mma (bf16 x bf16 -> fp32) into one of two TMEM accumulators;
//    warps 2..9 run the epilogue of tile i while the MMA of tile i+1 fills the
//    other accumulator ([ComFuse] PingPong MainLoop/Epilogue overlap).
//  * Epilogue = chained stage DAGs ([ComFuse] Stage-Stream Execution Model):
//    pass 1 streams 32-column fragments out of TMEM through the elementwise
//    nodes and aggregates thread-locally at the reduction node; the stage-1
//    value is written back into TMEM (the bypass path of Fig. 3, so GELU and
//    the bias are not recomputed); the reduce phase runs three levels
//    (thread-local over the fragment -> the other half-row's warps through
//    one shared-memory buffer -> the cluster over DSMEM with TMA bulk copies,
//    peer all-to-all for few CTAs or leader-follower for many) and, for wide
//    rows, the global partial buffer; pass 2 (the PostOp) re-reads TMEM,
//    normalises with the broadcast statistics and stores bf16.
//  * Every wait is bounded by %globaltimer; on expiry the error word in the
//    workspace records CF_ERR_DEVICE_TIMEOUT and all roles drain.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/cf.h"
#include "cf_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"
#include "trace.cuh"
#include "umma.cuh"

namespace cf {
namespace {

constexpr int kThreads = 320;      // 10 warps
constexpr int kEpiWarps = 8;       // warps 2..9: two groups of 4
constexpr int kGroupWarps = 4;     // one group: all 128 TMEM lanes (rows) of a tile
constexpr int kGroupThreads = 128;
constexpr int kBK = 64;            // K per stage (128 bytes of bf16: one swizzle atom)
constexpr int kABytes = kBlockM * kBK * 2;  // 16 KB

// named barriers (0 is __syncthreads): 1 + g for epilogue group g

// error info codes for the bounded pipeline waits
constexpr uint32_t kInfoProducer = 0x10000000u;
constexpr uint32_t kInfoMma = 0x20000000u;
constexpr uint32_t kInfoEpi = 0x30000000u;
constexpr uint32_t kInfoXchg = 0x40000000u;
constexpr uint32_t kInfoGlobal = 0x50000000u;

struct SmemLayout {
    uint32_t stage_bytes;  // A + B of one stage
    uint32_t ring;         // offset of the operand ring (1024-aligned)
    uint32_t stg;          // bf16 output staging, 1 or 2 x 2 KiB per epilogue warp (64B swizzle)
    uint32_t slot;         // float2 [sets][partials][128]: the row group's partials (4 x C, or 2 x 2C for a wide tile)
    uint32_t res;          // float2 [4][128]: leader-follower result, by exchange set
    uint32_t prm;          // float [2][3][256]: bias, gamma, beta of the tile's columns, per group
    uint32_t bars;         // mbarriers
    uint32_t total;        // bytes from the aligned base
};

constexpr int kXSets = 4;  // exchange buffer sets (tile mod 4)

__host__ __device__ inline SmemLayout smem_layout(int stages, int cluster, int n_slice, bool pair, bool leader,
                                                  int stg_bufs) {
    SmemLayout L;
    // a CTA of a pair stages its own 128 rows of X and half of the tile's W columns
    L.stage_bytes = kABytes + uint32_t(pair ? n_slice / 2 : n_slice) * kBK * 2;
    L.ring = 0;
    uint32_t off = L.ring + uint32_t(stages) * L.stage_bytes;
    L.stg = off;
    off += kEpiWarps * 2048 * uint32_t(stg_bufs);
    // exchange buffers exist only when a row group has more than one partial:
    // 4 sets x C (PingPong), or 2 sets x 2C for a wide tile (two groups per CTA,
    // one accumulator, so the CTAs of a cluster are never two tiles apart)
    const bool wide = n_slice > 256;
    const uint32_t xc = (cluster > 1 || wide) ? 1u : 0u;
    L.slot = off;
    off += xc * kXSets * uint32_t(cluster) * 128 * 8;
    L.res = off;  // the leader-follower result (not used by peer all-to-all)
    off += (leader ? xc : 0u) * kXSets * 128 * 8;
    L.prm = off;
    off += 2 * 3 * 256 * 4;
    L.bars = off;
    off += 256;
    L.total = off;
    return L;
}

// barrier slots inside L.bars (8 bytes each)
struct Bars {
    uint32_t full0, empty0;            // [stages] each
    uint32_t tmem_full0, tmem_empty0;  // [2]
    uint32_t xfull0, xres0;            // [kXSets]
    uint32_t mma_done;
    uint32_t misc;  // u32: tmem base, u32: abort flag
};

__device__ __forceinline__ Bars bars_at(uint32_t base, int stages) {
    Bars b;
    b.full0 = base;
    b.empty0 = base + 8 * stages;
    b.tmem_full0 = base + 16 * stages;
    b.tmem_empty0 = b.tmem_full0 + 16;
    b.xfull0 = b.tmem_empty0 + 16;
    b.xres0 = b.xfull0 + 8 * kXSets;
    b.mma_done = b.xres0 + 8 * kXSets;
    b.misc = b.mma_done + 8;
    return b;
}

// Softmax stage-1 nodes on one 32-column fragment, in base-2 units:
// t = acc * (alpha log2 e) + bias log2 e (p holds bias log2 e); online
// (max, sum 2^(t - max)) update; the fragment is replaced by 2^(t - m) where m
// is the running max after this fragment.  kMask: only the first `nvalid`
// columns take part (the rest are -inf, exp 0); a thread with no kept column
// so far keeps (m, s) = (-inf, 0).
template <bool kMask>
__device__ __forceinline__ void softmax_fragment(uint32_t (&v)[32], const float *p, float aL, float &m,
                                                 float &ssum, int nvalid = 32) {
    float t[32];
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
        const float4 b = *reinterpret_cast<const float4 *>(p + 4 * j4);
        ptx::fma2(t[4 * j4 + 0], t[4 * j4 + 1], __uint_as_float(v[4 * j4 + 0]), __uint_as_float(v[4 * j4 + 1]), aL,
                  aL, b.x, b.y);
        ptx::fma2(t[4 * j4 + 2], t[4 * j4 + 3], __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3]), aL,
                  aL, b.z, b.w);
    }
    if constexpr (kMask) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j >= nvalid) t[j] = neg_inf();
    }
    // fragment max: a tree of three-input maxima (17 instructions for 32 values)
    float c[11];
#pragma unroll
    for (int i = 0; i < 10; ++i) c[i] = ptx::max3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
    c[10] = fmaxf(t[30], t[31]);
    const float cm = ptx::max3(ptx::max3(c[0], c[1], c[2]), ptx::max3(c[3], c[4], c[5]),
                               ptx::max3(c[6], c[7], fmaxf(c[8], fmaxf(c[9], c[10]))));
    const float mn = fmaxf(m, cm);
    if (kMask && mn == neg_inf()) {  // nothing kept yet in this row slice
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
        return;
    }
    // exponentials and their sum two at a time (packed fp32 pairs, two partial sums)
    float sa = ssum * ptx::ex2_approx(m - mn), sb = 0.f;  // m = -inf on the first fragment: stays 0
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float d0, d1;
        ptx::add2(d0, d1, t[j], t[j + 1], -mn, -mn);
        const float e0 = ptx::ex2_approx(d0), e1 = ptx::ex2_approx(d1);  // masked: 2^-inf = 0
        ptx::add2(sa, sb, sa, sb, e0, e1);
        v[j] = __float_as_uint(e0);
        v[j + 1] = __float_as_uint(e1);
    }
    ssum = sa + sb;
    m = mn;
}

// LayerNorm stage-1 nodes on one fragment: x = alpha*acc + bias (-> GELU);
// the fragment is replaced by the stage-1 value; returns its (mean, M2).
// (With a residual: `r` holds the fragment's 32 bf16 residual values of this
// thread's row, added after the activation.)  Packed fp32 pairs throughout;
// the sums run in four independent chains.
template <bool kGelu>
__device__ __forceinline__ MeanM2 ln_fragment(uint32_t (&v)[32], const float *p, float alpha, const uint4 *r) {
    float x[32];
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
        const float4 b = *reinterpret_cast<const float4 *>(p + 4 * j4);
        ptx::fma2(x[4 * j4 + 0], x[4 * j4 + 1], __uint_as_float(v[4 * j4 + 0]), __uint_as_float(v[4 * j4 + 1]), alpha,
                  alpha, b.x, b.y);
        ptx::fma2(x[4 * j4 + 2], x[4 * j4 + 3], __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3]), alpha,
                  alpha, b.z, b.w);
    }
    if constexpr (kGelu) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) gelu_tanh_pair(x[j], x[j + 1]);
    }
    if (r != nullptr) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const uint4 q = r[j >> 3];
            const uint32_t w = ((j >> 1) & 3) == 0 ? q.x : ((j >> 1) & 3) == 1 ? q.y : ((j >> 1) & 3) == 2 ? q.z : q.w;
            ptx::add2(x[j], x[j + 1], x[j], x[j + 1], __uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        }
    }
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        v[j] = __float_as_uint(x[j]);
        v[j + 1] = __float_as_uint(x[j + 1]);
        v[j + 2] = __float_as_uint(x[j + 2]);
        v[j + 3] = __float_as_uint(x[j + 3]);
        ptx::add2(s0, s1, s0, s1, x[j], x[j + 1]);
        ptx::add2(s2, s3, s2, s3, x[j + 2], x[j + 3]);
    }
    const float mean = ((s0 + s1) + (s2 + s3)) * (1.0f / 32.0f);
    float q0 = 0.f, q1 = 0.f, q2 = 0.f, q3 = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        float d0, d1, d2, d3;
        ptx::add2(d0, d1, x[j], x[j + 1], -mean, -mean);
        ptx::add2(d2, d3, x[j + 2], x[j + 3], -mean, -mean);
        ptx::fma2(q0, q1, d0, d1, d0, d1, q0, q1);
        ptx::fma2(q2, q3, d2, d3, d2, d3, q2, q3);
    }
    return MeanM2{mean, (q0 + q1) + (q2 + q3)};
}

// Fold n (<= kN) partials p[0..n) of equal column count `cnt` in a fixed
// pairwise tree over index order (level W merges p[i] and p[i+W]); every CTA
// folding the same partials obtains bitwise-equal statistics.  The levels are
// compile-time so that p stays in registers.
template <bool kSoftmax, int kN, int W>
__device__ __forceinline__ void tree_level(float2 (&p)[kN], int n, float cnt) {
#pragma unroll
    for (int i = 0; i < kN; i += 2 * W) {
        const int nb = min(max(n - i - W, 0), W);  // p[i+W] covers nb partials; p[i] covers W
        if (nb > 0) {
            if constexpr (kSoftmax) {
                const MaxSum m = combine_maxsum(MaxSum{p[i].x, p[i].y}, MaxSum{p[i + W].x, p[i + W].y});
                p[i] = make_float2(m.m, m.s);
            } else {
                const MeanM2 m = combine_counts(MeanM2{p[i].x, p[i].y}, float(W) * cnt, MeanM2{p[i + W].x, p[i + W].y},
                                                float(nb) * cnt);
                p[i] = make_float2(m.mean, m.m2);
            }
        }
    }
    if constexpr (2 * W < kN) tree_level<kSoftmax, kN, 2 * W>(p, n, cnt);
}
template <bool kSoftmax, int kN>
__device__ __forceinline__ float2 tree_fold(float2 (&p)[kN], int n, float cnt) {
    tree_level<kSoftmax, kN, 1>(p, n, cnt);
    return p[0];
}

// The n (<= 16) partials of one row in the exchange slots (partial j at s[j*128]).
template <bool kSoftmax>
__device__ __forceinline__ float2 combine_slots(const float2 *s, int n, float cnt) {
    float2 p[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) p[j] = (j < n) ? s[j * 128] : make_float2(0.f, 0.f);
    return tree_fold<kSoftmax, 16>(p, n, cnt);
}

template <int EPI, bool kPair>
__global__ void __launch_bounds__(kThreads, 1) gemm_fused_kernel(const __grid_constant__ GemmArgs a, int stages) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    uint8_t *const gbase = smem_raw;
    // The 128B-swizzled operand tiles need a 1024-byte aligned ring.  The
    // dynamic shared window starts aligned; if it ever did not, report it and
    // do nothing (every CTA sees the same base, so none enters a cluster barrier).
    // A wide tile's two groups cannot share the global path: the host never plans
    // that; refuse it the same way.
    if ((base & 1023u) != 0u || (a.n_slice > 256 && a.groups > 1)) {
        ptx::griddep_wait();
        if (threadIdx.x == 0) ptx::record_error(a.err, 8u /*CF_ERR_DEVICE_BOUNDS*/, 0x60000000u | (base & 1023u));
        return;
    }

    constexpr bool kMask = EPI == EPI_SOFTMAX_MASK;        // causally masked softmax
    constexpr bool kSm = EPI == EPI_SOFTMAX || kMask;       // a softmax epilogue
    const int C = a.cluster;                // C_N: CTAs of one row group
    const int CM = kPair ? 2 : 1;           // row blocks per cluster
    const int G = a.groups;
    const int ns = a.n_slice;
    // a wide tile (512 columns) takes both accumulators and both epilogue groups
    const bool wide = !kPair && EPI != EPI_STORE_F32 && ns > 256;
    const int nk = a.K / kBK;
    const int T = a.super_blocks * G;       // tickets: (super row block, cluster group), row-block major
    const int nbox = ns / 64;               // 64-column W boxes of a tile
    const int my_boxes = kPair ? nbox / 2 : nbox;  // W boxes staged in this CTA
    const SmemLayout L = smem_layout(stages, C, ns, kPair, a.leader != 0, a.stg_bufs);
    const Bars B = bars_at(base + L.bars, stages);
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(gbase + (B.misc - base));
    volatile uint32_t *abort = misc + 1;
    const uint64_t tmo = a.timeout_ns;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t cid = ptx::cluster_id_x();
    const uint32_t ncl = ptx::nclusters_x();
    // Cluster rank = rank * C_M + m_sub: m_sub is this CTA's row block within the
    // cluster; a CTA pair (cta_group::2) is two consecutive ranks; `rank` is the
    // column slice within the row group {j * C_M + m_sub}.
    const int m_sub = int(crank) % CM;
    const uint32_t rank = crank / uint32_t(CM);
    const uint32_t pair_leader = crank & ~1u;         // even CTA of the pair (issues the MMAs)
    const bool is_leader = !kPair || (crank & 1u) == 0u;
    const uint32_t tmem_cols = wide ? 512u : (ns * 2 <= 32) ? 32u : uint32_t(ns * 2);
    const unsigned long long t_start = ptx::globaltimer();  // traced after the dependency wait
    // this thread arrived on the cluster barrier that ends the kernel (early: once no
    // peer can touch this CTA's shared memory any more)
    bool arrived = false;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(B.full0 + 8 * s, 1);
            ptx::mbar_init(B.empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(B.tmem_full0 + 8 * b, 1);
            // one epilogue group (4 warps) drains each accumulator; the pair
            // leader waits for both CTAs' groups; a wide tile, for both groups
            ptx::mbar_init(B.tmem_empty0 + 8 * b, kPair ? 2 * kGroupWarps : wide ? kEpiWarps : kGroupWarps);
        }
        for (int x = 0; x < kXSets; ++x) {
            ptx::mbar_init(B.xfull0 + 8 * x, 1);
            ptx::mbar_init(B.xres0 + 8 * x, 1);
        }
        ptx::mbar_init(B.mma_done, 1);
        misc[1] = 0u;
        ptx::fence_mbarrier_init_cluster();
    }
    if (warp == 1) {
        if constexpr (kPair) {
            ptx::tmem_alloc_pair(B.misc, tmem_cols);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(B.misc, tmem_cols);
            ptx::tmem_relinquish();
        }
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&a.tmap_x);
        ptx::prefetch_tensormap(&a.tmap_w);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // barrier initialisation is visible cluster-wide before any peer signals it
    ptx::cluster_sync();
    const uint32_t tmem_base = misc[0];
    // Programmatic dependent launch: the set-up above overlapped the previous
    // grid's tail; nothing in global memory is touched before it completed.
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (threadIdx.x == 0 && a.trace != nullptr) {
        a.trace[blockIdx.x * CF_TRACE_SLOTS + 0] = t_start;
        trace_stamp(a.trace, 1);
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // bytes landing on the full barrier of this CTA (pair: the leader's
            // barrier receives both CTAs' tiles)
            const uint32_t tx_cta = uint32_t(kABytes) + uint32_t(my_boxes) * 8192u;
            const uint32_t tx = kPair ? 2u * tx_cta : tx_cta;
            // W tiles are reused by every row block: keep them in L2 ahead of the
            // streaming output
            const uint64_t pol_w = ptx::policy_evict_last();
            uint32_t it = 0;         // k-blocks issued
            uint32_t s = 0, ph = 0;  // their ring position
            bool ok = true;
            int ptile = 0;
            for (int t = cid; t < T && ok; t += ncl, ++ptile) {
                const int rb = (t / G) * CM + m_sub, g = t % G;
                const int m0 = rb * kBlockM;
                const int n0 = (g * C + int(rank)) * ns;
                for (int kb = 0; kb < nk; ++kb) {
                    // every CTA that reads this stage has released it
                    ok = ptx::mbar_wait_bounded(B.empty0 + 8 * s, ph ^ 1u, tmo, abort, a.err, kInfoProducer | s);
                    if (!ok) break;
                    const uint32_t sa = base + L.ring + s * L.stage_bytes;
                    const uint32_t sb = sa + kABytes;
                    const uint32_t fb = B.full0 + 8 * s;
                    if constexpr (kPair) {
                        // both CTAs' loads complete on the leader's full barrier
                        const uint32_t fbl = ptx::mapa(fb, pair_leader);
                        if (is_leader) ptx::mbar_arrive_expect_tx(fb, tx);
                        ptx::tma_load_2d_pair(sa, &a.tmap_x, fbl, kb * kBK, m0);
                        // this CTA stages W columns [m_sub * ns/2, +ns/2) of the 256-row MMA's N:
                        // my_boxes 64-column blocks in one 3-D copy
                        ptx::tma_load_3d_pair_hint(sb, &a.tmap_w, fbl, 0, kb * kBK, n0 / 64 + m_sub * my_boxes, pol_w);
                    } else {
                        ptx::mbar_arrive_expect_tx(fb, tx);
                        ptx::tma_load_2d(sa, &a.tmap_x, fb, kb * kBK, m0);
                        ptx::tma_load_3d_hint(sb, &a.tmap_w, fb, 0, kb * kBK, n0 / 64, pol_w);  // nbox blocks
                    }
                    if (kb == 0) trace_tile(a.trace, ptile, CF_TR_TMA_FIRST);
                    if (kb == nk - 1) trace_tile(a.trace, ptile, CF_TR_TMA_LAST);
                    ++it;
                    if (++s == uint32_t(stages)) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // drain: every stage this producer filled has been released by all of
            // its readers (so every load landed and every release signal aimed at
            // this CTA arrived) before the CTA may exit
            const uint32_t issued = it;
            const uint32_t first = issued > uint32_t(stages) ? issued - uint32_t(stages) : 0u;
            for (uint32_t i = first; i < issued; ++i) {
                const uint32_t s = i % uint32_t(stages);
                const uint32_t ph = (i / uint32_t(stages)) & 1u;
                volatile uint32_t local_abort = 0;
                ptx::mbar_wait_bounded(B.empty0 + 8 * s, ph, tmo, &local_abort, nullptr, 0);
            }
        }
        __syncwarp();
        if constexpr (!kPair) {  // a single CTA's producer touches no peer's shared memory
            ptx::cluster_arrive_relaxed();
            arrived = true;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && is_leader) {
            // a wide tile is two N = 256 MMAs per K step into adjacent TMEM columns
            const uint32_t idesc = idesc_bf16(kPair ? 2 * kBlockM : kBlockM, wide ? 256 : ns);
            const uint16_t pair_mask = uint16_t(3u << pair_leader);
            // Operand descriptors of ring stage 0.  A stage's own are these plus its
            // byte offset >> 4 in the address field (the ring ends below 256 KB, so
            // the 14-bit field never carries); within a stage, A advances 16 K
            // elements = 32 B inside the swizzle atom and B (MN-major: 64-column
            // blocks 8 KB apart, 8-row K groups 1 KB apart) 16 K rows = 2 KB.  The
            // loop below keeps the single issuing thread's work between MMA groups
            // short, so the tensor pipe's queue never runs dry.
            const uint64_t ad0 = sw128_desc(base + L.ring, 16, 1024);
            const uint64_t bd0 = sw128_desc(base + L.ring + kABytes, 8192, 1024);
            uint32_t s = 0, ph = 0;  // ring position of the next k-block
            int tile = 0;
            for (int t = cid; t < T; t += ncl, ++tile) {
                const uint32_t buf = wide ? 0u : uint32_t(tile & 1);
                const uint32_t tph = wide ? (uint32_t(tile) & 1u) : ((uint32_t(tile) >> 1) & 1u);
                if (!ptx::mbar_wait_bounded(B.tmem_empty0 + 8 * buf, tph ^ 1u, tmo, abort, a.err, kInfoMma | buf))
                    break;
                trace_tile(a.trace, tile, CF_TR_MMA_ACC_FREE);
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + buf * uint32_t(ns);
                unsigned long long waited = 0;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    const uint32_t fb = B.full0 + 8 * s;
                    if (!ptx::mbar_try_wait(fb, ph)) {  // not landed yet: the bounded slow path
                        const unsigned long long w0 = a.trace ? ptx::globaltimer() : 0ull;
                        ok = ptx::mbar_wait_bounded(fb, ph, tmo, abort, a.err, kInfoMma | 0x100u | s);
                        if (!ok) break;
                        if (a.trace) waited += ptx::globaltimer() - w0;
                    }
                    if (kb == 0) trace_tile(a.trace, tile, CF_TR_MMA_FIRST);
                    ptx::tc_fence_after();
                    const uint64_t soff = uint64_t((s * L.stage_bytes) >> 4);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = ad0 + soff + uint64_t(2 * k);
                        const uint64_t bd = bd0 + soff + uint64_t(128 * k);
                        const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
                        if constexpr (kPair) {
                            ptx::mma_bf16_pair(d, ad, bd, idesc, accum);
                        } else {
                            ptx::mma_bf16(d, ad, bd, idesc, accum);
                            // wide: columns 256..511 from W blocks 4..7 (32 KB further)
                            if (wide) ptx::mma_bf16(d + 256u, ad, bd + uint64_t(32768 >> 4), idesc, accum);
                        }
                    }
                    // the stage is free once these MMAs completed (pair: in both CTAs)
                    if constexpr (kPair) ptx::mma_commit_pair_mc(B.empty0 + 8 * s, pair_mask);
                    else ptx::mma_commit(B.empty0 + 8 * s);
                    if (++s == uint32_t(stages)) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                // accumulator ready (pair: in both CTAs' tensor memory)
                if constexpr (kPair) ptx::mma_commit_pair_mc(B.tmem_full0 + 8 * buf, pair_mask);
                else ptx::mma_commit(B.tmem_full0 + 8 * buf);
                trace_tile(a.trace, tile, CF_TR_MMA_DONE);
                trace_tile_value(a.trace, tile, CF_TR_MMA_WAIT_NS, waited);
            }
            // every MMA issued has completed before TMEM may be released
            if constexpr (kPair) ptx::mma_commit_pair_mc(B.mma_done, uint16_t(1u << crank));
            else ptx::mma_commit(B.mma_done);
            volatile uint32_t local_abort = 0;
            ptx::mbar_wait_bounded(B.mma_done, 0, tmo, &local_abort, nullptr, 0);
        }
        __syncwarp();
        if constexpr (!kPair) {  // commits of a single CTA signal only its own barriers
            ptx::cluster_arrive_relaxed();
            arrived = true;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Two groups of 4 warps take alternate tiles (PingPong over the two TMEM
        // accumulators): while one group waits on an exchange or the global
        // barrier, the other streams its tile.  Warp w of a group reads TMEM
        // lane quadrant w % 4, so thread = one row, all n_slice columns.
        const int e = warp - 2;               // 0..7
        const int grp = e >> 2;               // epilogue group = accumulator buffer
        const int q = warp & 3;               // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;        // row of the tile == TMEM lane
        const int gt = (e & 3) * 32 + lane;   // thread index within the group
        const bool gt0 = (gt == 0);
        const uint32_t bar_grp = 1u + uint32_t(grp);
        float2 *const slot = reinterpret_cast<float2 *>(gbase + L.slot);
        float2 *const res = reinterpret_cast<float2 *>(gbase + L.res);
        float *const prm = reinterpret_cast<float *>(gbase + L.prm) + grp * 768;
        const uint32_t stg0 = base + L.stg + uint32_t(e) * 2048u * uint32_t(a.stg_bufs);  // this warp's staging
        uint32_t nstore = 0;  // stores issued by this warp (selects the staging buffer)
        const uint64_t pol_y = ptx::policy_evict_first();  // output is written once
        const float fN = float(a.N);
        const int ecols = wide ? 256 : ns;       // columns of a tile this group handles
        const int coff = wide ? grp * 256 : 0;   // and their offset within the tile
        const int nchunks = ecols / 32;          // 2, 4 or 8 fragments of 32 columns per thread
        const int parts = wide ? 2 : 1;  // partials per CTA: one per group on the tile
        const int npart = C * parts;     // partials of one row group
        float *const pb = prm;        // bias, gamma, beta of this group's current tile
        float *const pg = prm + 256;
        float *const pe = prm + 512;

        const int tstep = wide ? 1 : 2;  // PingPong: alternate tiles; wide: every tile
        int tile = wide ? 0 : grp;
        for (int t = cid + (wide ? 0 : grp) * ncl; t < T; t += tstep * ncl, tile += tstep) {
            const int rb = (t / G) * CM + m_sub, g = t % G;
            const int m0 = rb * kBlockM;
            const int ncta = (g * C + int(rank)) * ns + coff;  // first global column this group handles
            const uint32_t buf = wide ? 0u : uint32_t(grp);
            const uint32_t tph = wide ? (uint32_t(tile) & 1u) : ((uint32_t(tile) >> 1) & 1u);
            const uint32_t xs = wide ? (uint32_t(tile) & 1u) : (uint32_t(tile) & 3u);  // exchange buffer set
            const uint32_t xph = wide ? ((uint32_t(tile) >> 1) & 1u) : ((uint32_t(tile) >> 2) & 1u);

            // Row-vector parameters of the tile's columns into this group's shared
            // buffer, fetched before the accumulator is ready; the group's previous
            // tile finished reading them before the group barrier that ended it.
            if constexpr (EPI != EPI_STORE_F32) {
                for (int c = gt; c < ecols; c += kGroupThreads) {
                    pb[c] = a.bias ? __ldg(a.bias + ncta + c) * (kSm ? kLog2e : 1.f) : 0.f;
                    if constexpr (!kSm) {
                        pg[c] = __ldg(a.gamma + ncta + c);
                        pe[c] = a.beta ? __ldg(a.beta + ncta + c) : 0.f;
                    }
                }
            }
            ptx::mbar_wait_bounded(B.tmem_full0 + 8 * buf, tph, tmo, abort, a.err, kInfoEpi | buf);
            ptx::tc_fence_after();
            ptx::named_bar_sync(bar_grp, kGroupThreads);  // parameters visible to the group
            if (gt0) trace_tile(a.trace, tile, CF_TR_EPI_START);
            const uint32_t tacc = tmem_base + (uint32_t(q * 32) << 16) + buf * uint32_t(ns) + uint32_t(coff);

            if constexpr (EPI == EPI_STORE_F32) {
                // Unfused-baseline mode: the raw fp32 accumulator tile is written to
                // P [M, N]; no epilogue nodes, no row reduction.  Each 32-column
                // fragment leaves as two 16-column x 32-row blocks (64B swizzle).
                const bool rows_live = (m0 + q * 32) < a.M;
                const int ystore = m0 + q * 32;
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    if (c < nchunks) {
                        uint32_t v0[32], v1[32];
                        ptx::tmem_ld32(tacc + c * 32, v0);
                        ptx::tmem_ld32(tacc + (c + 1) * 32, v1);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t(&v)[32] = (k >> 1) == 0 ? v0 : v1;
                            const int hh = k & 1;
                            if (rows_live) {
                                const uint32_t stg = stg0 + (a.stg_bufs > 1 ? (nstore & 1u) * 2048u : 0u);
                                if (lane == 0) {
                                    if (a.stg_bufs > 1) ptx::bulk_wait_group_read1();
                                    else ptx::bulk_wait_group_read0();
                                }
                                __syncwarp();
                                const uint32_t ra = stg + uint32_t(lane) * 64u;
                                const uint32_t sw = (uint32_t(lane) >> 1) & 3u;
#pragma unroll
                                for (int k4 = 0; k4 < 4; ++k4)
                                    ptx::st_shared_v4(ra + ((uint32_t(k4) ^ sw) << 4), v[16 * hh + 4 * k4],
                                                      v[16 * hh + 4 * k4 + 1], v[16 * hh + 4 * k4 + 2],
                                                      v[16 * hh + 4 * k4 + 3]);
                                ptx::fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    ptx::tma_store_2d_hint(&a.tmap_y, stg, ncta + (c + (k >> 1)) * 32 + hh * 16, ystore, pol_y);
                                    ptx::bulk_commit_group();
                                }
                                ++nstore;
                            }
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (kPair) ptx::mbar_arrive_cluster(ptx::mapa(B.tmem_empty0 + 8 * buf, pair_leader));
                    else ptx::mbar_arrive(B.tmem_empty0 + 8 * buf);
                }
                ptx::named_bar_sync(bar_grp, kGroupThreads);
                continue;
            }

            // ---------------- stage 1: compute phase + thread-local aggregation.
            // Fragments of 32 columns stream out of TMEM two at a time; the stage-1
            // value is written back in place for the PostOp (bypass path).  The
            // thread's statistic covers the CTA's whole row slice.
            float2 part;     // LN: (mean, M2) over n_slice columns; softmax: (max, sum exp)
            float mrun[8];   // softmax: running max when each fragment's exps were taken
            if constexpr (kSm) {
                float m = neg_inf(), ssum = 0.f;
                // causal mask: columns of this row slice kept, counted from its first
                // column (clamped into each fragment below)
                const long long keep = kMask ? (long long)(m0 + row) + a.mask_offset - (long long)ncta + 1 : 0;
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    if (c < nchunks) {
                        uint32_t v0[32], v1[32];
                        ptx::tmem_ld32(tacc + c * 32, v0);
                        ptx::tmem_ld32(tacc + (c + 1) * 32, v1);
                        ptx::tmem_ld_wait();
                        const int nv0 = kMask ? int(keep - 32 * c < 0 ? 0 : keep - 32 * c > 32 ? 32 : keep - 32 * c) : 32;
                        const int nv1 = kMask ? int(keep - 32 * (c + 1) < 0 ? 0 : keep - 32 * (c + 1) > 32 ? 32
                                                                                                  : keep - 32 * (c + 1))
                                              : 32;
                        softmax_fragment<kMask>(v0, pb + c * 32, a.alpha * kLog2e, m, ssum, nv0);
                        mrun[c] = m;
                        ptx::tmem_st32(tacc + c * 32, v0);
                        softmax_fragment<kMask>(v1, pb + (c + 1) * 32, a.alpha * kLog2e, m, ssum, nv1);
                        mrun[c + 1] = m;
                        ptx::tmem_st32(tacc + (c + 1) * 32, v1);
                    }
                }
                ptx::tmem_st_wait();
                part = make_float2(m * kLn2, ssum);  // natural units for the exchange
            } else {
                MeanM2 acc{0.f, 0.f};
                // residual R [M, N] bf16: this thread's row slice of the fragment pair,
                // read (streaming) before the TMEM loads so the two latencies overlap
                const bool has_r = a.resid != nullptr;
                const uint4 *rrow = has_r && (m0 + row) < a.M
                                        ? reinterpret_cast<const uint4 *>(a.resid + size_t(m0 + row) * size_t(a.N) + ncta)
                                        : nullptr;
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    if (c < nchunks) {
                        uint32_t v0[32], v1[32];
                        uint4 r[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) r[k] = rrow ? __ldcs(rrow + c * 4 + k) : make_uint4(0u, 0u, 0u, 0u);
                        ptx::tmem_ld32(tacc + c * 32, v0);
                        ptx::tmem_ld32(tacc + (c + 1) * 32, v1);
                        ptx::tmem_ld_wait();
                        const MeanM2 c0 = ln_fragment<EPI == EPI_GELU_LN>(v0, pb + c * 32, a.alpha, has_r ? r : nullptr);
                        ptx::tmem_st32(tacc + c * 32, v0);
                        acc = (c == 0) ? c0 : combine_counts(acc, float(32 * c), c0, 32.f);
                        const MeanM2 c1 = ln_fragment<EPI == EPI_GELU_LN>(v1, pb + (c + 1) * 32, a.alpha,
                                                                          has_r ? r + 4 : nullptr);
                        ptx::tmem_st32(tacc + (c + 1) * 32, v1);
                        acc = combine_counts(acc, float(32 * (c + 1)), c1, 32.f);
                    }
                }
                ptx::tmem_st_wait();
                part = make_float2(acc.mean, acc.m2);
            }
            if (gt0) trace_tile(a.trace, tile, CF_TR_EPI_STATS);

            // ---------------- levels 2 and 3: a row's statistic over this CTA's columns
            // is one thread's (a wide tile: two threads', one per group).  Each thread
            // sends its row's partial straight into the gathering CTAs' shared memory
            // with an 8-byte st.async that completes on their mbarrier: every CTA of
            // the row group (peer all-to-all) or rank 0 (leader-follower, which sends
            // the combined statistics back with a bulk copy).  The gatherer folds
            // the partials in index order (CTA rank, then group), the same in every
            // CTA.  No shared-memory fence or group barrier precedes the sends.
            if (gt0) trace_tile(a.trace, tile, CF_TR_EPI_CTA);
            const bool lead_grp = !wide || grp == 0;  // does the per-CTA steps of the tile
            float2 stat;                              // row-group statistic of this row
            if (npart == 1) {
                stat = part;  // the row group is this CTA's one group
            } else if (!*abort) {
                const uint32_t xfull = B.xfull0 + 8 * xs;
                const uint32_t sl = base + L.slot + xs * uint32_t(npart) * 1024u;  // [npart][128] float2
                // this partial's index: CTA rank, then (wide tile) the group
                const uint32_t mine = sl + uint32_t(int(rank) * parts + (wide ? grp : 0)) * 1024u + uint32_t(row) * 8u;
                const float2 *slot_row = slot + size_t(xs) * size_t(npart) * 128u + row;
                if (!a.leader) {
                    if (gt0 && lead_grp) ptx::mbar_arrive_expect_tx(xfull, uint32_t(npart) * 1024u);
                    for (int r = 0; r < C; ++r) {
                        const uint32_t peer = uint32_t(r * CM + m_sub);
                        ptx::st_async_f2(ptx::mapa(mine, peer), part.x, part.y, ptx::mapa(xfull, peer));
                    }
                    ptx::mbar_wait_bounded<true>(xfull, xph, tmo, abort, a.err, kInfoXchg | xs);
                    stat = combine_slots<kSm>(slot_row, npart, float(ecols));
                } else {
                    if (gt0 && lead_grp) {
                        if (rank == 0) ptx::mbar_arrive_expect_tx(xfull, uint32_t(npart) * 1024u);
                        else ptx::mbar_arrive_expect_tx(B.xres0 + 8 * xs, 1024u);
                    }
                    ptx::st_async_f2(ptx::mapa(mine, uint32_t(m_sub)), part.x, part.y, ptx::mapa(xfull, uint32_t(m_sub)));
                    if (rank == 0) {
                        ptx::mbar_wait_bounded<true>(xfull, xph, tmo, abort, a.err, kInfoXchg | xs);
                        stat = combine_slots<kSm>(slot_row, npart, float(ecols));
                        if (lead_grp) {
                            res[xs * 128 + row] = stat;
                            ptx::fence_proxy_async_smem();
                            ptx::named_bar_sync(bar_grp, kGroupThreads);
                            if (gt0 && !*abort) {
                                const uint32_t src = base + L.res + xs * 1024;
                                for (int r = 1; r < C; ++r)
                                    ptx::bulk_copy_s2cluster(ptx::mapa(src, r * CM + m_sub), src, 1024,
                                                             ptx::mapa(B.xres0 + 8 * xs, r * CM + m_sub));
                            }
                        }
                    } else {
                        ptx::mbar_wait_bounded<true>(B.xres0 + 8 * xs, xph, tmo, abort, a.err, kInfoXchg | 0x10u | xs);
                        stat = res[xs * 128 + row];
                    }
                }
            } else {
                stat = part;  // aborting: the values no longer matter
            }
            if (gt0) trace_tile(a.trace, tile, CF_TR_EPI_CLUSTER);
            // After the group's last exchange no peer writes into this CTA's shared
            // memory again (every partial and result aimed at it has landed), and
            // every write of this thread into a peer has landed before that peer's
            // own wait passed: arrive on the final cluster barrier now, so the CTA
            // need not wait for its peers' stores at the end.  (Not after an abort,
            // where a wait may have given up with a partial still in flight.)
            if constexpr (!kPair) {
                if (!arrived && t + tstep * int(ncl) >= T && __all_sync(0xffffffffu, *abort == 0u)) {
                    ptx::cluster_arrive_relaxed();
                    arrived = true;
                }
            }

            // ---------------- level 4: rows wider than a cluster (global partials).
            // Layout [row block][g][128 rows] float2: one cluster group's 128 partials
            // are contiguous, so both the writes and each warp's reads are coalesced
            // 256-byte accesses.  After the last cluster's arrival
            // the critical path is three L2 round trips: its release arrive, the
            // pollers' acquire load that sees the full count, and one batch of
            // independent loads of all partials (up to 32 per batch).  The
            // error word is polled every 64 spins only, and this CTA's departure
            // (which lets the last one reset the counters) is taken off the path.
            uint32_t dep_old = 0;
            uint32_t *dep = nullptr;
            if (G > 1) {
                uint32_t *cnt = a.counters + rb;
                dep = a.counters + a.row_blocks_alloc + rb;
                const int Gp = G + (G & 1);
                float2 *pblk = a.partials + size_t(rb) * size_t(Gp) * 128u;
                if (rank == 0) {
                    pblk[g * 128 + row] = stat;
                    // the 128 writes happen before the barrier; the release arrive
                    // below publishes all of them
                    ptx::named_bar_sync(bar_grp, kGroupThreads);
                    if (gt0) ptx::red_add_release_gpu(cnt, 1u);
                }
                if (gt0) {
                    const uint32_t target = uint32_t(G + a.extra_arrivals);
                    const uint64_t t0 = ptx::globaltimer();
                    for (uint32_t spin = 0; !*abort; ++spin) {
                        if (ptx::ld_acquire_gpu(cnt) >= target) break;
                        if ((spin & 63u) == 63u && ptx::ld_relaxed_gpu(a.err) != 0u) {
                            *abort = 1u;
                            break;
                        }
                        if (ptx::globaltimer() - t0 > tmo) {
                            *abort = 1u;
                            ptx::record_error(a.err, 7u, kInfoGlobal | uint32_t(rb));
                            break;
                        }
                    }
                    // departure: the last of the row block's G * C CTAs resets its
                    // counters.  Relaxed: it is ordered after the acquire poll above
                    // (so every poll of the row block precedes the last departure),
                    // and nothing here waits for its result, looked at after pass 2.
                    dep_old = ptx::atom_add_relaxed_gpu(dep, 1u);
                }
                ptx::named_bar_sync(bar_grp, kGroupThreads);
                // combine in a fixed pairwise tree over index order (batches of 32, then
                // batch results left to right): every CTA of the row folds the same
                // partials identically, so all of them hold bitwise-equal statistics
                const float nc = float(ns * C);  // columns behind each partial
                float2 s2 = make_float2(0.f, 0.f);
                float sn = 0.f;
                for (int g0 = 0; g0 < G; g0 += 32) {
                    const int rem = G - g0;  // partials in this batch (>= 1; <= 32 used)
                    float2 p[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        p[i] = (i < rem) ? ptx::ld_relaxed_gpu_f2(pblk + (g0 + i) * 128 + row) : make_float2(0.f, 0.f);
                    tree_fold<kSm, 32>(p, rem, nc);
                    const float bn = float(min(rem, 32)) * nc;
                    if (g0 == 0) {
                        s2 = p[0];
                    } else if constexpr (kSm) {
                        const MaxSum m = combine_maxsum(MaxSum{s2.x, s2.y}, MaxSum{p[0].x, p[0].y});
                        s2 = make_float2(m.m, m.s);
                    } else {
                        const MeanM2 m = combine_counts(MeanM2{s2.x, s2.y}, sn, MeanM2{p[0].x, p[0].y}, bn);
                        s2 = make_float2(m.mean, m.m2);
                    }
                    sn += bn;
                }
                stat = s2;
            }
            if (gt0) trace_tile(a.trace, tile, CF_TR_EPI_GLOBAL);

            // ---------------- stage 2 (PostOp): broadcast the statistic back over the row,
            // bf16 into this warp's staging buffer, TMA bulk store of each 32x32 block
            const bool rows_live = (m0 + q * 32) < a.M;  // warp-uniform: this warp's 32 rows exist
            const int ystore = m0 + q * 32;
            float mean = 0.f, rstd = 0.f;
            if constexpr (!kSm) {
                // LayerNorm: (g - mean) / sqrt(M2/N + eps); RMSNorm: g / sqrt(mean(g^2) + eps)
                // with mean(g^2) = M2/N + mean^2 from the same statistics
                const float var = stat.y / fN;
                mean = a.rms ? 0.f : stat.x;
                rstd = rsqrtf((a.rms ? fmaf(stat.x, stat.x, var) : var) + a.eps);
            }
#pragma unroll
            for (int c = 0; c < 8; c += 2) {
                if (c < nchunks) {
                    uint32_t v0[32], v1[32];
                    ptx::tmem_ld32(tacc + c * 32, v0);
                    ptx::tmem_ld32(tacc + (c + 1) * 32, v1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        uint32_t(&v)[32] = k == 0 ? v0 : v1;
                        const int cc = c + k;
                        uint32_t w[16];
                        if constexpr (kSm) {
                            // a fully masked row (sum 0) is all zeros
                            const float f =
                                (kMask && !(stat.y > 0.f)) ? 0.f : ptx::ex2_approx(mrun[cc] - stat.x * kLog2e) / stat.y;
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                w[j] = ptx::pack_bf16x2(__uint_as_float(v[2 * j]) * f, __uint_as_float(v[2 * j + 1]) * f);
                        } else {
                            const float *gp = pg + cc * 32;
                            const float *bp = pe + cc * 32;
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                const float4 gm = *reinterpret_cast<const float4 *>(gp + 4 * j4);
                                const float4 bt = *reinterpret_cast<const float4 *>(bp + 4 * j4);
                                float d0, d1, d2, d3;  // (g - mean) rstd, then * gamma + beta, on pairs
                                ptx::add2(d0, d1, __uint_as_float(v[4 * j4 + 0]), __uint_as_float(v[4 * j4 + 1]), -mean, -mean);
                                ptx::add2(d2, d3, __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3]), -mean, -mean);
                                ptx::mul2(d0, d1, d0, d1, rstd, rstd);
                                ptx::mul2(d2, d3, d2, d3, rstd, rstd);
                                ptx::fma2(d0, d1, d0, d1, gm.x, gm.y, bt.x, bt.y);
                                ptx::fma2(d2, d3, d2, d3, gm.z, gm.w, bt.z, bt.w);
                                w[2 * j4] = ptx::pack_bf16x2(d0, d1);
                                w[2 * j4 + 1] = ptx::pack_bf16x2(d2, d3);
                            }
                        }
                        if (rows_live) {
                            // the previous store from this buffer has finished reading it
                            // (with two buffers: at most one store may still be reading)
                            const uint32_t stg = stg0 + (a.stg_bufs > 1 ? (nstore & 1u) * 2048u : 0u);
                            if (lane == 0) {
                                if (a.stg_bufs > 1) ptx::bulk_wait_group_read1();
                                else ptx::bulk_wait_group_read0();
                            }
                            __syncwarp();
                            // row `lane` of the 32x32 block: four 16-byte pieces, 64B swizzle
                            const uint32_t ra = stg + uint32_t(lane) * 64u;
                            const uint32_t sw = (uint32_t(lane) >> 1) & 3u;
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)
                                ptx::st_shared_v4(ra + ((uint32_t(k4) ^ sw) << 4), w[4 * k4], w[4 * k4 + 1],
                                                  w[4 * k4 + 2], w[4 * k4 + 3]);
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                ptx::tma_store_2d_hint(&a.tmap_y, stg, ncta + cc * 32, ystore, pol_y);
                                ptx::bulk_commit_group();
                            }
                            ++nstore;
                        }
                    }
                }
            }
            // accumulator buffer free for the MMA of tile + 2 (pair: tell the leader)
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kPair) ptx::mbar_arrive_cluster(ptx::mapa(B.tmem_empty0 + 8 * buf, pair_leader));
                else ptx::mbar_arrive(B.tmem_empty0 + 8 * buf);
            }
            // the group's shared parameters may be rewritten for its next tile only
            // after every thread of the group is done with them
            ptx::named_bar_sync(bar_grp, kGroupThreads);
            if (gt0) trace_tile(a.trace, tile, CF_TR_EPI_STORED);
            // the last CTA of the row block to depart resets its counters (for the
            // next launch on this workspace); every poller of this launch is done
            if (gt0 && dep != nullptr && dep_old == uint32_t(G * C) - 1u) {
                ptx::st_relaxed_gpu(a.counters + rb, 0u);
                ptx::st_relaxed_gpu(dep, 0u);
            }
        }
        // every bulk store of this warp has finished reading its staging buffer
        // before the CTA may leave (the writes complete with the grid)
        if (lane == 0) ptx::bulk_wait_group_read0();
        __syncwarp();
    }
    if (threadIdx.x == 64) trace_stamp(a.trace, 2);

    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // no CTA leaves while a peer may still access its shared memory
    if (!arrived) ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
    if (warp == 1) {
        if constexpr (kPair) ptx::tmem_dealloc_pair(tmem_base, tmem_cols);
        else ptx::tmem_dealloc(tmem_base, tmem_cols);
    }
    if (threadIdx.x == 64) trace_stamp(a.trace, 3);
}

void *kernel_for(int kind, bool pair) {
    switch (kind) {
        case EPI_STORE_F32:
            return pair ? reinterpret_cast<void *>(&gemm_fused_kernel<EPI_STORE_F32, true>)
                        : reinterpret_cast<void *>(&gemm_fused_kernel<EPI_STORE_F32, false>);
        case EPI_LN:
            return pair ? reinterpret_cast<void *>(&gemm_fused_kernel<EPI_LN, true>)
                        : reinterpret_cast<void *>(&gemm_fused_kernel<EPI_LN, false>);
        case EPI_GELU_LN:
            return pair ? reinterpret_cast<void *>(&gemm_fused_kernel<EPI_GELU_LN, true>)
                        : reinterpret_cast<void *>(&gemm_fused_kernel<EPI_GELU_LN, false>);
        case EPI_SOFTMAX:
            return pair ? reinterpret_cast<void *>(&gemm_fused_kernel<EPI_SOFTMAX, true>)
                        : reinterpret_cast<void *>(&gemm_fused_kernel<EPI_SOFTMAX, false>);
        case EPI_SOFTMAX_MASK:
            return pair ? reinterpret_cast<void *>(&gemm_fused_kernel<EPI_SOFTMAX_MASK, true>)
                        : reinterpret_cast<void *>(&gemm_fused_kernel<EPI_SOFTMAX_MASK, false>);
        default: return nullptr;
    }
}

// Function attributes are set once per (device, kernel) to the largest
// shared-memory size seen, so launches made under stream capture issue no
// attribute calls.
cudaError_t ensure_attributes(int variant, void *fn, int smem) {
    static int set_smem[64][16] = {};
    static bool nonportable[64][16] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || variant < 0 || variant >= 16) return cudaErrorInvalidValue;
    if (smem > set_smem[dev][variant]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        set_smem[dev][variant] = smem;
    }
    if (!nonportable[dev][variant]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        nonportable[dev][variant] = true;
    }
    return cudaSuccess;
}

}  // namespace

int gemm_fused_smem_bytes(int stages, int cluster, int n_slice, bool pair, bool leader, int stg_bufs) {
    return int(smem_layout(stages, cluster, n_slice, pair, leader, stg_bufs).total);
}

int gemm_fused_max_active_clusters(int kind, bool pair, int cluster, int smem) {
    void *fn = kernel_for(kind, pair);
    if (!fn) return 0;
    if (ensure_attributes(kind * 2 + (pair ? 1 : 0), fn, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster * 64);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_gemm_fused(int kind, const GemmArgs &a, int clusters, int stages, int smem, bool pdl,
                              cudaStream_t stream) {
    const bool pair = a.cluster_m == 2;
    void *fn = kernel_for(kind, pair);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = ensure_attributes(kind * 2 + (pair ? 1 : 0), fn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(clusters * a.cluster * a.cluster_m);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.cluster * a.cluster_m;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    int st = stages;
    void *args[] = {(void *)&a, (void *)&st};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace cf
