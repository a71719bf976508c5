// b2b.cu -- back-to-back GEMM with the intermediate kept on chip:
//     O = S . W2,   S = F(alpha * X.W1 + b1) in bf16,   F = row softmax or GELU
// ([ComFuse] B2BGEMM, Eqs. 3-7, Fig. 5); F = row softmax, GELU(tanh) or row
// LayerNorm over the N1 columns.
//
// Design (sm_103a):
//  * A cluster of C CTAs takes one 128-row block at a time; CTA rank r owns
//    the 256 columns [256 r, 256 r + 256) of the intermediate P = X.W1 (the
//    output space of MatMul_1 is partitioned along N1, Fig. 5).
//  * ML_1: tcgen05.mma accumulates P_tile (128 x 256, fp32) in tensor memory.
//  * Epi_1: F over P_tile.  For softmax (max, sum exp) and LayerNorm
//    (mean, M2) the row statistics are reduced over the cluster: every thread
//    sends its row's partial to each CTA with an 8-byte st.async.  S_tile = F(P_tile) is written back to
//    tensor memory as packed bf16 over the first 128 (consumed) columns of
//    P, so S never leaves the SM (Eq. 3 keeps it in registers; tcgen05.mma
//    reads a register-like A operand from tensor memory instead).
//  * ML_2: tcgen05.mma with A = S_tile from tensor memory and B = the CTA's
//    256-row slice of W2, streamed through the same operand ring as X and W1
//    (one multi-stage buffer for both MatMuls, Eq. 6); each CTA accumulates
//    its partial O_tile^(c) = S_tile^(c) W2^(c) (Eq. 4) into the second half
//    of the tile's tensor-memory columns.
//  * Epi_2: the partials are summed over the cluster (Eq. 5) as a
//    reduce-scatter: CTA r owns output columns [r N2/C, (r+1) N2/C); every
//    CTA sends each owner its partial columns with 16-byte st.async, and the
//    owner adds them in rank order (deterministic), rounds to bf16, stores.
//  * Every CTA loads the whole X tile itself from L2: sharing one copy
//    across the cluster would couple the CTAs' operand rings (a slot is
//    refilled only when all C MMAs released it).
//  * Two epilogue groups (4 warps each, one row per thread) own 256 tensor-
//    memory columns each and take alternate tiles, staggered by one stage
//    (Eq. 7): while one group runs Epi_1 / Epi_2, the MMA warp runs the other
//    group's ML_1 / ML_2.  MMA issue order: ML_1(0), then per tile t
//    ML_1(t+1), ML_2(t); the producer fills the ring in the same order.
//  * Every wait is bounded by %globaltimer; a timeout records
//    CF_ERR_DEVICE_TIMEOUT in the workspace error word and the roles drain.
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

constexpr int kThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2..5 group 0, warps 6..9 group 1
constexpr int kN1Slice = 256;   // columns of P per CTA
constexpr int kBK = 64;         // K per stage
constexpr int kABytes = 128 * kBK * 2;           // X tile: 16 KB
constexpr int kWBytes = kBK * kN1Slice * 2;      // W1 tile: 32 KB (a W2 tile uses N2*128 B of it)
constexpr int kStageBytes = kABytes + kWBytes;   // 48 KB

constexpr uint32_t kInfoProducer = 0x81000000u;
constexpr uint32_t kInfoMma = 0x82000000u;
constexpr uint32_t kInfoEpi = 0x83000000u;

struct Layout {
    uint32_t ring, slot, recv, prm, bars, total;
};

__host__ __device__ inline Layout layout(int stages, int C, int N2, int op) {
    Layout L;
    L.ring = 0;
    uint32_t off = uint32_t(stages) * kStageBytes;
    L.slot = off;  // float2 [2 groups][C][128]: softmax partials
    off += 2u * uint32_t(C) * 128u * 8u;
    L.recv = off;  // float4 [C][N2 / C / 4][128]: the partial output columns this CTA owns
                   // (row fastest, so a warp's 32 rows fill 512 consecutive bytes)
    off += 128u * uint32_t(N2) * 4u;
    L.prm = off;   // float [256] b1 (LayerNorm F: [3][256] b1, gamma1, beta1) of this CTA's columns
    off += (op == 2 ? 3u : 1u) * kN1Slice * 4u;
    L.bars = off;
    off += 256;
    L.total = off;
    return L;
}

// mbarriers; the per-group ones are pairs (group g at +8 g)
struct Bars {
    uint32_t full0, empty0, p_full, s_full, o_full, acc_free, xfull, rbar, rfree, mma_done, misc;
};
__device__ __forceinline__ Bars bars_at(uint32_t b, int stages) {
    Bars r;
    r.full0 = b;
    r.empty0 = b + 8 * stages;
    r.p_full = b + 16 * stages;
    r.s_full = r.p_full + 16;
    r.o_full = r.s_full + 16;
    r.acc_free = r.o_full + 16;
    r.xfull = r.acc_free + 16;
    r.rbar = r.xfull + 16;
    r.rfree = r.rbar + 16;
    r.mma_done = r.rfree + 16;
    r.misc = r.mma_done + 8;  // u32 tmem base, u32 abort flag
    return r;
}

template <int OP, int kN2>  // OP: 0 softmax, 1 GELU, 2 LayerNorm; kN2: 64 or 128
__global__ void __launch_bounds__(kThreads, 1) b2b_kernel(const __grid_constant__ B2bArgs a, int stages) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    if ((base & 1023u) != 0u) {
        ptx::griddep_wait();
        if (threadIdx.x == 0) ptx::record_error(a.err, 8u /*CF_ERR_DEVICE_BOUNDS*/, 0x60000000u | (base & 1023u));
        return;
    }
    const int C = a.cluster;
    const int w = kN2 / C;  // output columns owned by each CTA
    const int nk1 = (a.K + kBK - 1) / kBK;  // a ragged last block reads zeros past K
    constexpr int nk2 = kN1Slice / kBK;     // 4
    const Layout L = layout(stages, C, kN2, OP);
    const Bars B = bars_at(base + L.bars, stages);
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem_raw + (B.misc - base));
    volatile uint32_t *abort = misc + 1;
    const uint64_t tmo = a.timeout_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t cid = ptx::cluster_id_x();
    const uint32_t ncl = ptx::nclusters_x();
    const int RB = (a.M + 127) / 128;
    // tiles of this cluster: row blocks cid, cid + ncl, ...
    const int T = int(cid) < RB ? (RB - int(cid) + int(ncl) - 1) / int(ncl) : 0;
    unsigned long long *const tr = a.trace;
    const unsigned long long t_start = ptx::globaltimer();

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(B.full0 + 8 * s, 1);
            ptx::mbar_init(B.empty0 + 8 * s, 1);
        }
        for (int g = 0; g < 2; ++g) {
            ptx::mbar_init(B.p_full + 8 * g, 1);
            ptx::mbar_init(B.s_full + 8 * g, 4);
            ptx::mbar_init(B.o_full + 8 * g, 1);
            ptx::mbar_init(B.acc_free + 8 * g, 4);
            ptx::mbar_init(B.xfull + 8 * g, 1);
            ptx::mbar_init(B.rbar + 8 * g, 1);
            ptx::mbar_init(B.rfree + 8 * g, 4u * uint32_t(C));
        }
        ptx::mbar_init(B.mma_done, 1);
        misc[1] = 0u;
        ptx::fence_mbarrier_init_cluster();
    }
    if (warp == 1) {
        ptx::tmem_alloc(B.misc, 512);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&a.tmap_x);
        ptx::prefetch_tensormap(&a.tmap_w1);
        ptx::prefetch_tensormap(&a.tmap_w2);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_sync();
    const uint32_t tmem = misc[0];  // group g: columns [256 g, 256 g + 256)
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (threadIdx.x == 0 && tr != nullptr) {
        tr[blockIdx.x * CF_TRACE_SLOTS + 0] = t_start;
        trace_stamp(tr, 1);
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_last();
            uint32_t s = 0, ph = 0, it = 0;
            bool ok = true;
            auto next = [&]() {
                ++it;
                if (++s == uint32_t(stages)) {
                    s = 0;
                    ph ^= 1u;
                }
            };
            auto load_ml1 = [&](int t) {  // MatMul_1: X and this CTA's W1 columns
                const int m0 = (int(cid) + t * int(ncl)) * 128;
                for (int kb = 0; kb < nk1 && ok; ++kb) {
                    ok = ptx::mbar_wait_bounded(B.empty0 + 8 * s, ph ^ 1u, tmo, abort, a.err, kInfoProducer | s);
                    if (!ok) break;
                    if (kb == 0) trace_tile(tr, t, CF_TRB_TMA_FIRST);
                    const uint32_t sa = base + L.ring + s * kStageBytes, fb = B.full0 + 8 * s;
                    ptx::mbar_arrive_expect_tx(fb, uint32_t(kStageBytes));
                    ptx::tma_load_2d(sa, &a.tmap_x, fb, kb * kBK, m0);
                    ptx::tma_load_3d_hint(sa + kABytes, &a.tmap_w1, fb, 0, kb * kBK, int(rank) * (kN1Slice / 64),
                                          pol_w);
                    next();
                }
            };
            auto load_ml2 = [&]() {  // MatMul_2: this CTA's 256-row slice of W2, 64 rows per stage
                for (int kb = 0; kb < nk2 && ok; ++kb) {
                    ok = ptx::mbar_wait_bounded(B.empty0 + 8 * s, ph ^ 1u, tmo, abort, a.err, kInfoProducer | s);
                    if (!ok) break;
                    const uint32_t sa = base + L.ring + s * kStageBytes, fb = B.full0 + 8 * s;
                    ptx::mbar_arrive_expect_tx(fb, uint32_t(kBK) * uint32_t(kN2) * 2u);
                    ptx::tma_load_3d_hint(sa + kABytes, &a.tmap_w2, fb, 0, int(rank) * kN1Slice + kb * kBK, 0,
                                          pol_w);
                    next();
                }
            };
            if (T > 0) load_ml1(0);
            for (int t = 0; t < T && ok; ++t) {
                if (t + 1 < T) load_ml1(t + 1);
                load_ml2();
            }
            // every stage filled has been released before the CTA may exit
            const uint32_t first = it > uint32_t(stages) ? it - uint32_t(stages) : 0u;
            for (uint32_t i = first; i < it; ++i) {
                volatile uint32_t local_abort = 0;
                ptx::mbar_wait_bounded(B.empty0 + 8 * (i % uint32_t(stages)), (i / uint32_t(stages)) & 1u, tmo,
                                       &local_abort, nullptr, 0);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id1 = idesc_bf16(128, kN1Slice);
            const uint32_t id2 = idesc_bf16(128, kN2);  // A from tensor memory (K-major), B = W2 MN-major
            const uint64_t ad0 = sw128_desc(base + L.ring, 16, 1024);
            const uint64_t bd0 = sw128_desc(base + L.ring + kABytes, 8192, 1024);
            uint32_t s = 0, ph = 0;
            bool ok = true;
            auto stage_ready = [&](uint32_t info) -> bool {
                if (ptx::mbar_try_wait(B.full0 + 8 * s, ph)) return true;
                return ptx::mbar_wait_bounded(B.full0 + 8 * s, ph, tmo, abort, a.err, info | s);
            };
            auto release = [&]() {
                ptx::mma_commit(B.empty0 + 8 * s);
                if (++s == uint32_t(stages)) {
                    s = 0;
                    ph ^= 1u;
                }
            };
            auto ml1 = [&](int t) {
                const int g = t & 1;
                const uint32_t dP = tmem + uint32_t(256 * g);
                for (int kb = 0; kb < nk1; ++kb) {
                    ok = stage_ready(kInfoMma);
                    if (!ok) return;
                    if (kb == 0) trace_tile(tr, t, CF_TRB_ML1_FIRST);
                    ptx::tc_fence_after();
                    const uint64_t soff = uint64_t((s * uint32_t(kStageBytes)) >> 4);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        ptx::mma_bf16(dP, ad0 + soff + uint64_t(2 * k), bd0 + soff + uint64_t(128 * k), id1,
                                      (kb | k) != 0 ? 1u : 0u);
                    release();
                }
                ptx::mma_commit(B.p_full + 8 * g);
                trace_tile(tr, t, CF_TRB_ML1_DONE);
            };
            auto ml2 = [&](int t) {
                const int g = t & 1;
                const uint32_t tg = tmem + uint32_t(256 * g);
                trace_tile(tr, t, CF_TRB_ML2_START);
                // O^(c) = S^(c) W2^(c): K = 256 in four 64-deep stages; per MMA,
                // K = 16 bf16 of A = 8 tensor-memory columns
                for (int kb = 0; kb < nk2; ++kb) {
                    ok = stage_ready(kInfoMma | 0x300u);
                    if (!ok) return;
                    ptx::tc_fence_after();
                    const uint64_t soff = uint64_t((s * uint32_t(kStageBytes)) >> 4);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        ptx::mma_bf16_ts(tg + 128u, tg + uint32_t(kb * 32 + k * 8), bd0 + soff + uint64_t(128 * k),
                                         id2, (kb | k) != 0 ? 1u : 0u);
                    release();
                }
                ptx::mma_commit(B.o_full + 8 * g);
                trace_tile(tr, t, CF_TRB_ML2_DONE);
            };
            if (T > 0) ml1(0);
            for (int t = 0; t < T && ok; ++t) {
                if (t + 1 < T) {
                    // the columns of tile t+1's group are free once Epi_2 of tile t-1 read its O
                    const int u = t + 1;
                    ok = ptx::mbar_wait_bounded(B.acc_free + 8 * (u & 1), ((u >> 1) & 1) ^ 1, tmo, abort, a.err,
                                                kInfoMma | 0x100u);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    ml1(u);
                    if (!ok) break;
                }
                ok = ptx::mbar_wait_bounded(B.s_full + 8 * (t & 1), (t >> 1) & 1, tmo, abort, a.err,
                                            kInfoMma | 0x200u);
                if (!ok) break;
                ptx::tc_fence_after();
                ml2(t);
            }
            ptx::mma_commit(B.mma_done);
            volatile uint32_t local_abort = 0;
            ptx::mbar_wait_bounded(B.mma_done, 0, tmo, &local_abort, nullptr, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue groups
        const int g = (warp - 2) >> 2;
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;
        const bool lead = (warp == 2 + 4 * g) && lane == 0;
        const uint32_t tg = tmem + uint32_t(256 * g) + (uint32_t(q * 32) << 16);
        float *const prm = reinterpret_cast<float *>(smem_raw + L.prm);
        const float2 *slot = reinterpret_cast<const float2 *>(smem_raw + L.slot) + size_t(g) * size_t(C) * 128u;
        const float4 *recv = reinterpret_cast<const float4 *>(smem_raw + L.recv);
        const int w4 = w / 4;
        const int n0 = int(rank) * kN1Slice;
        for (int c = threadIdx.x - 64; c < kN1Slice; c += 256) {
            prm[c] = a.b1 ? __ldg(a.b1 + n0 + c) : 0.f;
            if constexpr (OP == 2) {
                prm[kN1Slice + c] = __ldg(a.gamma1 + n0 + c);
                prm[2 * kN1Slice + c] = __ldg(a.beta1 + n0 + c);
            }
        }
        ptx::named_bar_sync(1, 256);
        for (int t = g, j = 0; t < T; t += 2, ++j) {
            const uint32_t par = uint32_t(j) & 1u;
            const int m0 = (int(cid) + t * int(ncl)) * 128;
            if (!ptx::mbar_wait_bounded(B.p_full + 8 * g, par, tmo, abort, a.err, kInfoEpi | g)) break;
            ptx::tc_fence_after();
            if (lead) trace_tile(tr, t, CF_TRB_EPI1_START);
            // ---------------- Epi_1: S = F(alpha * P + b1), bf16 into the group's first 128 columns
            if constexpr (OP == 0) {
                float m = neg_inf(), ssum = 0.f, mrun[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tg + c * 32, v);
                    ptx::tmem_ld_wait();
                    float cm = neg_inf();
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float z = fmaf(a.alpha, __uint_as_float(v[k]), prm[c * 32 + k]);
                        v[k] = __float_as_uint(z);
                        cm = fmaxf(cm, z);
                    }
                    const float mn = fmaxf(m, cm);
                    float s = ssum * ptx::ex2_approx((m - mn) * kLog2e);
                    const float off = mn * kLog2e;
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float e = ptx::ex2_approx(fmaf(__uint_as_float(v[k]), kLog2e, -off));
                        s += e;
                        v[k] = __float_as_uint(e);
                    }
                    ssum = s;
                    m = mn;
                    mrun[c] = mn;
                    ptx::tmem_st32(tg + c * 32, v);
                }
                ptx::tmem_st_wait();
                if (lead) trace_tile(tr, t, CF_TRB_EPI1_LOCAL);
                // row statistics over the cluster: every thread sends its row's
                // (max, sum) to each CTA; the gatherers fold them in rank order
                const uint32_t xb = B.xfull + 8 * g;
                float2 st = make_float2(m, ssum);
                if (C > 1 && !*abort) {
                    if (lead) ptx::mbar_arrive_expect_tx(xb, uint32_t(C) * 1024u);
                    const uint32_t mine = base + L.slot + (uint32_t(g) * uint32_t(C) + rank) * 1024u + uint32_t(row) * 8u;
                    for (int r = 0; r < C; ++r)
                        ptx::st_async_f2(ptx::mapa(mine, uint32_t(r)), m, ssum, ptx::mapa(xb, uint32_t(r)));
                    if (!ptx::mbar_wait_bounded<true>(xb, par, tmo, abort, a.err, kInfoEpi | 0x10u | g)) break;
                    st = slot[row];
                    for (int r = 1; r < C; ++r) {
                        const float2 o = slot[r * 128 + row];
                        const MaxSum mm = combine_maxsum(MaxSum{st.x, st.y}, MaxSum{o.x, o.y});
                        st = make_float2(mm.m, mm.s);
                    }
                }
                const float inv = 1.0f / st.y;
                // S = exp(z - m_row) / s_row, packed bf16 over the consumed P columns
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32], sv[16];
                    ptx::tmem_ld32(tg + c * 32, v);
                    ptx::tmem_ld_wait();
                    const float f = ptx::ex2_approx((mrun[c] - st.x) * kLog2e) * inv;
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        sv[k] = ptx::pack_bf16x2(__uint_as_float(v[2 * k]) * f, __uint_as_float(v[2 * k + 1]) * f);
                    ptx::tmem_st16(tg + c * 16, sv);
                }
            } else if constexpr (OP == 2) {
                // pass 1: z = alpha * P + b1 back into tensor memory; (mean, M2) of
                // the row slice, two passes per 32-column fragment, folded by counts
                MeanM2 acc{0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32];
                    float z[32];
                    ptx::tmem_ld32(tg + c * 32, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        z[k] = fmaf(a.alpha, __uint_as_float(v[k]), prm[c * 32 + k]);
                        v[k] = __float_as_uint(z[k]);
                    }
                    const MeanM2 cm = chunk_mean_m2(z);
                    acc = c == 0 ? cm : combine_counts(acc, float(32 * c), cm, 32.f);
                    ptx::tmem_st32(tg + c * 32, v);
                }
                ptx::tmem_st_wait();
                if (lead) trace_tile(tr, t, CF_TRB_EPI1_LOCAL);
                // row statistics over the cluster (every CTA holds 256 of the row's
                // N1 values): each thread sends its (mean, M2) to every CTA, the
                // gatherers fold them in rank order
                const uint32_t xb = B.xfull + 8 * g;
                MeanM2 st = acc;
                if (C > 1 && !*abort) {
                    if (lead) ptx::mbar_arrive_expect_tx(xb, uint32_t(C) * 1024u);
                    const uint32_t mine = base + L.slot + (uint32_t(g) * uint32_t(C) + rank) * 1024u + uint32_t(row) * 8u;
                    for (int r = 0; r < C; ++r)
                        ptx::st_async_f2(ptx::mapa(mine, uint32_t(r)), acc.mean, acc.m2, ptx::mapa(xb, uint32_t(r)));
                    if (!ptx::mbar_wait_bounded<true>(xb, par, tmo, abort, a.err, kInfoEpi | 0x10u | g)) break;
                    st = MeanM2{slot[row].x, slot[row].y};
                    for (int r = 1; r < C; ++r) {
                        const float2 o = slot[r * 128 + row];
                        st = combine_counts(st, float(kN1Slice * r), MeanM2{o.x, o.y}, float(kN1Slice));
                    }
                }
                const float rstd = rsqrtf(st.m2 / float(kN1Slice * C) + a.eps);
                // pass 2: S = (z - mean) * rstd * gamma1 + beta1, packed bf16
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32], sv[16];
                    ptx::tmem_ld32(tg + c * 32, v);
                    ptx::tmem_ld_wait();
                    const float *ga = prm + kN1Slice + c * 32, *be = prm + 2 * kN1Slice + c * 32;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float y0 = fmaf((__uint_as_float(v[2 * k]) - st.mean) * rstd, ga[2 * k], be[2 * k]);
                        const float y1 =
                            fmaf((__uint_as_float(v[2 * k + 1]) - st.mean) * rstd, ga[2 * k + 1], be[2 * k + 1]);
                        sv[k] = ptx::pack_bf16x2(y0, y1);
                    }
                    ptx::tmem_st16(tg + c * 16, sv);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32], sv[16];
                    ptx::tmem_ld32(tg + c * 32, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float x0 = gelu_tanh_dev(fmaf(a.alpha, __uint_as_float(v[2 * k]), prm[c * 32 + 2 * k]));
                        const float x1 =
                            gelu_tanh_dev(fmaf(a.alpha, __uint_as_float(v[2 * k + 1]), prm[c * 32 + 2 * k + 1]));
                        sv[k] = ptx::pack_bf16x2(x0, x1);
                    }
                    ptx::tmem_st16(tg + c * 16, sv);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(B.s_full + 8 * g);
            if (lead) trace_tile(tr, t, CF_TRB_EPI1_DONE);
            // ---------------- Epi_2: reduce-scatter of the partial outputs over the cluster
            if (!ptx::mbar_wait_bounded(B.o_full + 8 * g, par, tmo, abort, a.err, kInfoEpi | 0x20u | g)) break;
            ptx::tc_fence_after();
            if (lead) trace_tile(tr, t, CF_TRB_EPI2_START);
            uint32_t o[kN2 / 32][32];
#pragma unroll
            for (int c = 0; c < kN2 / 32; ++c) ptx::tmem_ld32(tg + 128u + c * 32, o[c]);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(B.acc_free + 8 * g);  // ML_1 of tile t+2 may overwrite the columns
            const uint32_t rb = B.rbar + 8 * g;
            if (lead) ptx::mbar_arrive_expect_tx(rb, 128u * uint32_t(kN2) * 4u);
            // every owner has read the previous tile's partials out of its buffer
            if (t > 0 && !ptx::mbar_wait_bounded<true>(B.rfree + 8 * ((t - 1) & 1), ((t - 1) >> 1) & 1, tmo, abort,
                                                       a.err, kInfoEpi | 0x28u | g))
                break;
            if (!*abort) {
#pragma unroll
                for (int c = 0; c < kN2 / 32; ++c) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        const int col = c * 32 + k;
                        const int owner = col / w, kk = col % w;
                        const uint32_t dst = base + L.recv +
                                             ((rank * uint32_t(w4) + uint32_t(kk >> 2)) * 128u + uint32_t(row)) * 16u;
                        ptx::st_async_f4(ptx::mapa(dst, uint32_t(owner)), __uint_as_float(o[c][k]),
                                         __uint_as_float(o[c][k + 1]), __uint_as_float(o[c][k + 2]),
                                         __uint_as_float(o[c][k + 3]), ptx::mapa(rb, uint32_t(owner)));
                    }
                }
            }
            if (lead) trace_tile(tr, t, CF_TRB_EPI2_SENT);
            if (!ptx::mbar_wait_bounded<true>(rb, par, tmo, abort, a.err, kInfoEpi | 0x30u | g)) break;
            if (lead) trace_tile(tr, t, CF_TRB_EPI2_RECV);
            // O[row, rank*w .. +w) = sum over the cluster, in rank order
            if (m0 + row < a.M) {
                uint16_t *orow = a.out + size_t(m0 + row) * size_t(kN2) + size_t(rank) * size_t(w);
                for (int k0 = 0; k0 < w; k0 += 8) {
                    const int q0 = k0 >> 2;
                    float4 lo = recv[q0 * 128 + row], hi = recv[(q0 + 1) * 128 + row];
                    for (int r = 1; r < C; ++r) {
                        const float4 l2 = recv[(r * w4 + q0) * 128 + row], h2 = recv[(r * w4 + q0 + 1) * 128 + row];
                        lo.x += l2.x; lo.y += l2.y; lo.z += l2.z; lo.w += l2.w;
                        hi.x += h2.x; hi.y += h2.y; hi.z += h2.z; hi.w += h2.w;
                    }
                    uint4 ov;
                    ov.x = ptx::pack_bf16x2(lo.x, lo.y);
                    ov.y = ptx::pack_bf16x2(lo.z, lo.w);
                    ov.z = ptx::pack_bf16x2(hi.x, hi.y);
                    ov.w = ptx::pack_bf16x2(hi.z, hi.w);
                    *reinterpret_cast<uint4 *>(orow + k0) = ov;
                }
            }
            if (lead) trace_tile(tr, t, CF_TRB_EPI2_STORED);
            // this warp's rows of the buffer are free again: one arrival at every sender
            __syncwarp();
            if (lane == 0)
                for (int r = 0; r < C; ++r) ptx::mbar_arrive_cluster(ptx::mapa(B.rfree + 8 * g, uint32_t(r)));
        }
    }

    // ------------------------------------------------------------ teardown
    if (threadIdx.x == 64) trace_stamp(tr, 2);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_sync();  // no CTA leaves while a peer may still write its shared memory
    if (warp == 1) ptx::tmem_dealloc(tmem, 512);
    if (threadIdx.x == 64) trace_stamp(tr, 3);
}

template <int OP>
void *b2b_fn_n2(int n2) {
    return n2 == 64 ? reinterpret_cast<void *>(&b2b_kernel<OP, 64>) : reinterpret_cast<void *>(&b2b_kernel<OP, 128>);
}
void *b2b_fn(int op, int n2) {
    if (op == 0) return b2b_fn_n2<0>(n2);
    if (op == 1) return b2b_fn_n2<1>(n2);
    return b2b_fn_n2<2>(n2);
}

}  // namespace

int b2b_smem_bytes(int stages, int cluster, int n2, int op) { return int(layout(stages, cluster, n2, op).total); }

int b2b_max_active_clusters(int op, int cluster, int n2, int smem) {
    void *fn = b2b_fn(op, n2);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
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

cudaError_t launch_b2b(int op, const B2bArgs &a, int clusters, int stages, int smem, bool pdl, cudaStream_t stream) {
    void *fn = b2b_fn(op, a.N2);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(clusters * a.cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.cluster;
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
