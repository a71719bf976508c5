// b2b_stream.cu -- back-to-back GEMM with one CTA per 128-row block:
//     O = S . W2,   S = F(alpha * X.W1 + b1) in bf16,
//     F = row softmax, GELU or row LayerNorm (gamma1, beta1)
// ([ComFuse] B2BGEMM, Eqs. 3-7, Fig. 5), with the N1 columns of the
// intermediate streamed through tensor memory in 256-column chunks instead of
// being partitioned over a cluster.
//
// Design (sm_103a):
//  * A persistent CTA takes 128-row blocks in turn; the intermediate's N1
//    columns are chunks J of 256.  Tensor memory: S (256 fp32 columns,
//    ML_1's accumulator), P (128 columns: the chunk's bf16 values, packed in
//    pairs, ML_2's A operand) and O (N2 fp32 columns, ML_2's accumulator over
//    the row block's chunks).
//  * ML_1(J): S = X . W1[:, chunk J], one N = 256 MMA per K step (narrower
//    MMAs from shared-memory operands take about as long each).  X stays in
//    shared memory for the row block when K <= 128 (double-buffered across row
//    blocks); otherwise each k-block of X streams through the ring with W1's.
//  * Epi_1(J): four epilogue groups (4 warps each, one per TMEM lane quadrant;
//    thread = row) take 64 columns of the chunk each, so a thread holds 64
//    values (576 threads: 96 registers each).  Once S is in registers it may
//    be overwritten, so ML_1(J+1) starts while Epi_1(J) computes
//    z = alpha * S + b1 and F, and writes the bf16 values to P as soon as
//    ML_2(J-1) has read the previous ones.
//    Softmax is evaluated online (running max m and sum l per row, base-2
//    exponentials): the groups exchange their parts' row maxima through
//    shared memory; m is raised -- and O and l rescaled -- only when the
//    chunk's max exceeds it by more than 8 (a factor 256), so most chunks
//    leave O alone.
//    The values rounded to bf16 are these unnormalised exponentials (at most
//    256); the division by the row sum happens once, on the fp32 output.
//    LayerNorm in one pass: the row's shift mu0 is the mean of its first
//    chunk (the groups exchange their parts); each chunk feeds ML_2 with
//    (z - mu0) gamma1 and folds its (mean, M2) into the group's running pair;
//    the output is rstd O - rstd (mu - mu0) gamma1^T W2 + beta1^T W2, the two
//    rows from b2b_ln_fold_kernel (launched first; waited for only before the
//    first output stage).
//  * ML_2(J): O += P . W2[chunk J, :] (K = 256), A read from tensor memory.
//  * Issue order: ML_1(0), then ML_1(J+1), ML_2(J) for each J: the tensor
//    core runs ML_1(J+1) and ML_2(J-1) under Epi_1(J).
//  * End of a row block: O / l (GELU: O; LayerNorm: as above), group g
//    writing output columns [32 g, 32 g + 32) through a 2 KB staging buffer
//    per warp and 32 x 32 TMA stores (where X streams and F keeps row
//    statistics, directly from registers: that room is a fourth ring stage).
//    No cluster, no exchange with other CTAs.
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

constexpr int kGroups = 4;      // epilogue groups of 4 warps (one per TMEM lane quadrant)
constexpr int kThreads = 64 + 128 * kGroups;  // warp 0 TMA, warp 1 MMA, then the groups' warps
constexpr int kChunk = 256;     // N1 columns per chunk
constexpr int kCols = kChunk / kGroups;  // columns of a chunk one epilogue group handles (64)
constexpr int kFrag = kCols / 32;        // its 32-column fragments
constexpr int kBK = 64;         // K per k-block
constexpr int kXBlock = 128 * kBK * 2;       // one k-block of X: 16 KB
constexpr int kW1Block = kBK * kChunk * 2;   // one k-block of a W1 chunk: 32 KB
constexpr int kMaxResidentK = 128;           // X kept for the row block up to this K
constexpr float kRescale = 8.f;              // raise the running max only past 2^8
constexpr uint32_t kColP = 256, kColO = 384; // tensor-memory columns of P and O (S at 0)

constexpr uint32_t kInfoProducer = 0x91000000u;
constexpr uint32_t kInfoMma = 0x92000000u;
constexpr uint32_t kInfoEpi = 0x93000000u;

// Shared-memory layout, fixed per epilogue and mode (compile-time offsets keep
// the epilogue's registers for its data): resident X (K <= 128) with a
// 3-stage ring of 32 KB, or X streamed with W1 through a ring of 4 stages of
// 48 KB.  The output leaves through TMA stores from a staging buffer, except
// where X streams and the epilogue keeps row statistics (softmax, LayerNorm):
// there the fourth stage takes that room and each thread writes its row's
// 64-byte segments directly.
template <int OP, bool kRes>
__host__ __device__ constexpr bool direct_out() {
    return !kRes && OP != 1;
}

struct Layout {
    uint32_t xres, xbytes, ring, stage, stages, stg, bias, xm, stat, bars, total;
};

template <int OP, bool kRes>
__host__ __device__ constexpr Layout layout() {
    Layout L{};
    L.xres = 0;  // resident mode: X of two row blocks, two 16 KB k-blocks each
    L.xbytes = kRes ? 2u * kXBlock : 0u;
    L.ring = 2u * L.xbytes;  // 1024-aligned: every block above is a multiple of 16 KB
    // a stage holds a W1 k-block (and the X k-block when X streams), or half
    // of a W2 chunk (128 rows x N2 <= 32 KB)
    L.stage = kRes ? uint32_t(kW1Block) : uint32_t(kXBlock + kW1Block);
    // (GELU has no row statistics: a fourth stage fits when X streams)
    L.stages = kRes ? 3u : 4u;
    L.stg = L.ring + L.stages * L.stage;  // bf16 output staging: 2 KB (32 x 32, 64B swizzle) per epilogue warp
    // float [groups][2 chunk parities][kCols]: b1 of the group's columns (LayerNorm:
    // [groups][2][2][kCols], b1 and gamma1)
    L.bias = L.stg + (direct_out<OP, kRes>() ? 0u : 4u * kGroups * 2048u);
    L.xm = L.bias + kGroups * 2u * kCols * 4u * (OP == 2 ? 2u : 1u);
    // softmax: float [2 chunk parities][groups][128] row maxima; LayerNorm:
    // float [2 rb parities][groups][128] means of the row block's first chunk
    L.stat = L.xm + (OP != 1 ? 2u * kGroups * 128u * 4u : 0u);
    // softmax: float [2 rb parities][groups][128] row sums; LayerNorm: float2
    // [2 rb parities][groups][128] (mean, M2) of each group's columns
    L.bars = L.stat + (OP == 0 ? 2u * kGroups * 128u * 4u : OP == 2 ? 2u * kGroups * 128u * 8u : 0u);
    L.total = L.bars + 256u;
    return L;
}

struct Bars {
    uint32_t full0, empty0, xfull0, xfree0, s_full, s_free, p_full, o_full, mfree, mma_done, misc;
};
__device__ __forceinline__ Bars bars_at(uint32_t b, int stages) {
    Bars r;
    r.full0 = b;
    r.empty0 = b + 8 * stages;
    r.xfull0 = b + 16 * stages;  // [2] resident X buffers
    r.xfree0 = r.xfull0 + 16;    // [2]
    r.s_full = r.xfree0 + 16;    // ML_1 of the chunk complete
    r.s_free = r.s_full + 8;     // every group read S (all epilogue warps)
    r.p_full = r.s_free + 8;     // every group wrote P (all epilogue warps)
    r.o_full = r.p_full + 8;     // ML_2 of the chunk complete
    r.mfree = r.o_full + 8;      // the row block's output read O (all epilogue warps)
    r.mma_done = r.mfree + 8;
    r.misc = r.mma_done + 8;  // u32 tmem base, u32 abort flag
    return r;
}

template <int OP, int kN2, bool kDirect>
__device__ __forceinline__ void stream_output(const CUtensorMap *tmap_o, uint16_t *out, int M, int m0, uint32_t tO_group,
                                           uint32_t stg, float *st, float lk, MeanM2 ls, float mu0, const float *fold,
                                           float n1, float eps, int g, int q, int lane, uint32_t mfree,
                                           volatile uint32_t *abort, unsigned long long *stamp) {
    constexpr int kOut = 32;  // output columns of a group: groups 0 .. N2/32 - 1 write, the rest only sync
    const int row = q * 32 + lane;
    const uint32_t tO = tO_group + uint32_t(kOut * g);
    float inv = 1.f;
    if constexpr (OP == 0) {
        st[g * 128 + row] = lk;
        ptx::named_bar_sync(kGroups + 1, 128 * kGroups);
        float lsum = 0.f;
#pragma unroll
        for (int h = 0; h < kGroups; ++h) lsum += st[h * 128 + row];
        inv = 1.f / lsum;
    }
    // LayerNorm: O = rstd (sum_n (z_n - mu0) gamma1_n W2_nk) - rstd (mu - mu0) c1_k + c0_k,
    // c1 = gamma1^T W2 and c0 = beta1^T W2 (fold)
    float sh = 0.f;
    if constexpr (OP == 2) {
        ptx::griddep_wait();  // the fold kernel has completed (no-op after the first row block)
        float2 *const st2 = reinterpret_cast<float2 *>(st);
        st2[g * 128 + row] = make_float2(ls.mean, ls.m2);
        ptx::named_bar_sync(kGroups + 1, 128 * kGroups);
        const float ng = n1 * (1.f / float(kGroups));  // columns of a group
        MeanM2 rs{st2[row].x, st2[row].y};
#pragma unroll
        for (int h = 1; h < kGroups; ++h)
            rs = combine_counts(rs, ng * float(h), MeanM2{st2[h * 128 + row].x, st2[h * 128 + row].y}, ng);
        inv = rsqrtf(rs.m2 / n1 + eps);
        sh = (rs.mean - mu0) * inv;
    }
    if (g * kOut >= kN2) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(mfree);
        return;
    }
    const bool live = m0 + q * 32 < M && !*abort && out != nullptr;  // warp-uniform
    const uint32_t sw = (uint32_t(lane) >> 1) & 3u;
    const uint64_t pol_o = ptx::policy_evict_first();  // the output is written once
#pragma unroll
    for (int c = 0; c < kOut / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c * 32, o);
        ptx::tmem_ld_wait();
        if (c == kOut / 32 - 1) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(mfree);  // ML_2 of the next row block may overwrite O
        }
        if (live) {
            uint32_t w[16];
            if constexpr (OP == 2) {
                const int k0 = g * kOut + c * 32;
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const float2 c1 = __ldg(reinterpret_cast<const float2 *>(fold + k0) + h);
                    const float2 c0 = __ldg(reinterpret_cast<const float2 *>(fold + kN2 + k0) + h);
                    w[h] = ptx::pack_bf16x2(fmaf(__uint_as_float(o[2 * h]), inv, fmaf(-sh, c1.x, c0.x)),
                                            fmaf(__uint_as_float(o[2 * h + 1]), inv, fmaf(-sh, c1.y, c0.y)));
                }
            } else {
#pragma unroll
                for (int h = 0; h < 16; ++h)
                    w[h] = ptx::pack_bf16x2(__uint_as_float(o[2 * h]) * inv, __uint_as_float(o[2 * h + 1]) * inv);
            }
            if constexpr (kDirect) {
                // the row's 32 columns: 64 contiguous bytes
                if (m0 + row < M) {
                    uint4 *const dst =
                        reinterpret_cast<uint4 *>(out + size_t(m0 + row) * size_t(kN2) + size_t(g * kOut + c * 32));
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) dst[k4] = make_uint4(w[4 * k4], w[4 * k4 + 1], w[4 * k4 + 2], w[4 * k4 + 3]);
                }
                continue;
            }
            if (lane == 0) ptx::bulk_wait_group_read0();  // the previous store read the buffer
            __syncwarp();
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
                ptx::st_shared_v4(stg + uint32_t(lane) * 64u + ((uint32_t(k4) ^ sw) << 4), w[4 * k4], w[4 * k4 + 1],
                                  w[4 * k4 + 2], w[4 * k4 + 3]);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_2d_hint(tmap_o, stg, g * kOut + c * 32, m0 + q * 32, pol_o);
                ptx::bulk_commit_group();
            }
        }
    }
    if (stamp != nullptr && lane == 0) *stamp = ptx::globaltimer();
}

// OP: 0 softmax, 1 GELU, 2 LayerNorm; kN2: 64 or 128; kRes: X resident (K <= 128)
template <int OP, int kN2, bool kRes>
__global__ void __launch_bounds__(kThreads, 1) b2b_stream_kernel(const __grid_constant__ B2bArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    if ((base & 1023u) != 0u) {
        ptx::griddep_wait();
        if (threadIdx.x == 0) ptx::record_error(a.err, 8u /*CF_ERR_DEVICE_BOUNDS*/, 0x60000000u | (base & 1023u));
        return;
    }
    const int nk1 = (a.K + kBK - 1) / kBK;  // a ragged last block reads zeros past K
    constexpr bool resident = kRes;
    constexpr Layout L = layout<OP, kRes>();
    constexpr int stages = int(L.stages);
    const int nc = a.N1 / kChunk;           // chunks per row block
    const Bars B = bars_at(base + L.bars, stages);
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem_raw + (B.misc - base));
    volatile uint32_t *abort = misc + 1;
    const uint64_t tmo = a.timeout_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RB = (a.M + 127) / 128;
    // row blocks of this CTA: blockIdx.x, + gridDim.x, ...; chunks J = i * nc + j
    const int nrb = int(blockIdx.x) < RB ? (RB - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x) : 0;
    const int NJ = nrb * nc;
    unsigned long long *const tr = a.trace;
    const unsigned long long t_start = ptx::globaltimer();

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(B.full0 + 8 * s, 1);
            ptx::mbar_init(B.empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(B.xfull0 + 8 * b, 1);
            ptx::mbar_init(B.xfree0 + 8 * b, 1);
        }
        ptx::mbar_init(B.s_full, 1);
        ptx::mbar_init(B.s_free, 4 * kGroups);
        // (test hook: extra arrivals that never come make the MMA warp's wait
        // for P run out -- CF_ERR_DEVICE_TIMEOUT, every role drains)
        ptx::mbar_init(B.p_full, 4 * kGroups + uint32_t(a.extra_arrivals));
        ptx::mbar_init(B.o_full, 1);
        ptx::mbar_init(B.mfree, 4 * kGroups);
        ptx::mbar_init(B.mma_done, 1);
        misc[1] = 0u;
        ptx::fence_mbarrier_init_cluster();  // (a CTA is its own cluster of one)
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
    const uint32_t tmem = misc[0];
    ptx::griddep_launch_dependents();
    // LayerNorm: the fold kernel launched just before this one let it start
    // only once the grids before the fold had completed, so the inputs are
    // ready; the fold's own output is waited for before the first output stage
    if constexpr (OP != 2) ptx::griddep_wait();
    if (threadIdx.x == 0 && tr != nullptr) {
        tr[blockIdx.x * CF_TRACE_SLOTS + 0] = t_start;
        trace_stamp(tr, 1);
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Fills the ring in the MMA warp's consumption order: ML_1(0), then
        // ML_1(J+1), ML_2(J) for each J.
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_last();
            uint32_t s = 0, ph = 0, it = 0;
            bool ok = true;
            auto acquire = [&]() -> uint32_t {  // next free stage; returns its full barrier
                ok = ptx::mbar_wait_bounded(B.empty0 + 8 * s, ph ^ 1u, tmo, abort, a.err, kInfoProducer | s);
                return B.full0 + 8 * s;
            };
            auto next = [&]() {
                ++it;
                if (++s == uint32_t(stages)) {
                    s = 0;
                    ph ^= 1u;
                }
            };
            int i1 = 0, j1 = 0;  // (row block, chunk) of the next ML_1
            auto load_ml1 = [&](int J) {
                const int i = i1, j = j1;
                if (++j1 == nc) {
                    j1 = 0;
                    ++i1;
                }
                const int m0 = (int(blockIdx.x) + i * int(gridDim.x)) * 128;
                trace_tile(tr, J, CF_TRB_TMA_FIRST);
                if (resident && j == 0) {
                    // X of row block i into buffer i & 1, once row block i - 2 is done with it
                    const int b = i & 1;
                    if (i >= 2) {
                        ok = ptx::mbar_wait_bounded(B.xfree0 + 8 * b, uint32_t((i >> 1) - 1) & 1u, tmo, abort, a.err,
                                                    kInfoProducer | 0x100u);
                        if (!ok) return;
                    }
                    ptx::mbar_arrive_expect_tx(B.xfull0 + 8 * b, uint32_t(nk1) * uint32_t(kXBlock));
                    for (int kb = 0; kb < nk1; ++kb)
                        ptx::tma_load_2d(base + L.xres + uint32_t(b) * L.xbytes + uint32_t(kb) * kXBlock, &a.tmap_x,
                                         B.xfull0 + 8 * b, kb * kBK, m0);
                }
                for (int kb = 0; kb < nk1 && ok; ++kb) {
                    const uint32_t fb = acquire();
                    if (!ok) break;
                    const uint32_t sa = base + L.ring + s * L.stage;
                    if (resident) {
                        ptx::mbar_arrive_expect_tx(fb, uint32_t(kW1Block));
                        ptx::tma_load_3d_hint(sa, &a.tmap_w1, fb, 0, kb * kBK, j * (kChunk / 64), pol_w);
                    } else {
                        ptx::mbar_arrive_expect_tx(fb, uint32_t(kXBlock + kW1Block));
                        ptx::tma_load_2d(sa, &a.tmap_x, fb, kb * kBK, m0);
                        ptx::tma_load_3d_hint(sa + kXBlock, &a.tmap_w1, fb, 0, kb * kBK, j * (kChunk / 64), pol_w);
                    }
                    next();
                }
            };
            int j2 = 0;  // chunk of the next ML_2
            auto load_ml2 = [&](int J) {  // W2 rows [256 j, 256 j + 256) in two stages of 128
                const int j = j2;
                if (++j2 == nc) j2 = 0;
                for (int h = 0; h < 2 && ok; ++h) {
                    const uint32_t fb = acquire();
                    if (!ok) break;
                    const uint32_t sa = base + L.ring + s * L.stage;
                    ptx::mbar_arrive_expect_tx(fb, 128u * uint32_t(kN2) * 2u);
                    ptx::tma_load_3d_hint(sa, &a.tmap_w2, fb, 0, j * kChunk + h * 128, 0, pol_w);
                    next();
                }
            };
            if (NJ > 0) load_ml1(0);
            for (int J = 0; J < NJ && ok; ++J) {
                if (J + 1 < NJ) load_ml1(J + 1);
                load_ml2(J);
            }
            // every stage filled has been released before the CTA may exit
            const uint32_t first = it > uint32_t(stages) ? it - uint32_t(stages) : 0u;
            for (uint32_t k = first; k < it; ++k) {
                volatile uint32_t local_abort = 0;
                ptx::mbar_wait_bounded(B.empty0 + 8 * (k % uint32_t(stages)), (k / uint32_t(stages)) & 1u, tmo,
                                       &local_abort, nullptr, 0);
            }
            // and every resident X load landed (the MMA warp waited for them unless aborting)
            if (resident)
                for (int i = nrb > 2 ? nrb - 2 : 0; i < nrb; ++i) {
                    volatile uint32_t local_abort = 0;
                    ptx::mbar_wait_bounded(B.xfull0 + 8 * (i & 1), uint32_t(i >> 1) & 1u, tmo, &local_abort, nullptr,
                                           0);
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id1 = idesc_bf16(128, kChunk);
            const uint32_t id2 = idesc_bf16(128, kN2);  // A from tensor memory (K-major), B = W2 MN-major
            // X k-blocks: K-major, 128B swizzle; a W1 k-block: four 64-column
            // blocks 8 KB apart; a W2 half chunk: N2/64 blocks of 128 rows, 16 KB apart
            const uint64_t xd0 = sw128_desc(base + L.xres, 16, 1024);
            const uint64_t rd_x = sw128_desc(base + L.ring, 16, 1024);
            const uint64_t rd_w1 = sw128_desc(base + L.ring, 8192, 1024);
            const uint64_t rd_w2 = sw128_desc(base + L.ring, 16384, 1024);
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
            // (row block, chunk) of the next ML_1 and the next ML_2, advanced in
            // place: this thread's instructions between MMA groups are few (it
            // shares its SMSP's issue slots with four epilogue warps)
            int i1 = 0, j1 = 0, i2 = 0, j2 = 0;
            auto ml1 = [&](int J) {
                const int i = i1, j = j1;
                if (++j1 == nc) {
                    j1 = 0;
                    ++i1;
                }
                // S is free once both groups read the previous chunk
                if (J > 0) {
                    ok = ptx::mbar_wait_bounded(B.s_free, uint32_t(J - 1) & 1u, tmo, abort, a.err, kInfoMma | 0x100u);
                    if (!ok) return;
                }
                if (resident && j == 0) {
                    ok = ptx::mbar_wait_bounded(B.xfull0 + 8 * (i & 1), uint32_t(i >> 1) & 1u, tmo, abort, a.err,
                                                kInfoMma | 0x500u);
                    if (!ok) return;
                }
                trace_tile(tr, J, CF_TRB_ML1_FIRST);
                ptx::tc_fence_after();
                const uint64_t xd = xd0 + uint64_t(((uint32_t(i & 1) * L.xbytes)) >> 4);
                for (int kb = 0; kb < nk1; ++kb) {
                    ok = stage_ready(kInfoMma);
                    if (!ok) return;
                    ptx::tc_fence_after();
                    const uint64_t soff = uint64_t((s * L.stage) >> 4);
                    const uint64_t ad = resident ? xd + uint64_t((uint32_t(kb) * uint32_t(kXBlock)) >> 4) : rd_x + soff;
                    const uint64_t bd = rd_w1 + soff + (resident ? 0u : uint64_t(uint32_t(kXBlock) >> 4));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        ptx::mma_bf16(tmem, ad + uint64_t(2 * k), bd + uint64_t(128 * k), id1, (kb | k) != 0 ? 1u : 0u);
                    release();
                }
                if (resident && j == nc - 1) ptx::mma_commit(B.xfree0 + 8 * (i & 1));  // X buffer reusable
                ptx::mma_commit(B.s_full);
                trace_tile(tr, J, CF_TRB_ML1_DONE);
            };
            auto ml2 = [&](int J) {
                const int i = i2, j = j2;
                if (++j2 == nc) {
                    j2 = 0;
                    ++i2;
                }
                ok = ptx::mbar_wait_bounded(B.p_full, uint32_t(J) & 1u, tmo, abort, a.err, kInfoMma | 0x200u);
                if (!ok) return;
                // the row block's first ML_2 overwrites O: the previous row block's
                // output has read it
                if (j == 0 && i > 0) {
                    ok = ptx::mbar_wait_bounded(B.mfree, uint32_t(i - 1) & 1u, tmo, abort, a.err, kInfoMma | 0x300u);
                    if (!ok) return;
                }
                ptx::tc_fence_after();
                trace_tile(tr, J, CF_TRB_ML2_START);
                // K = 256 in sixteen steps of 16 bf16 = 8 packed tensor-memory
                // columns; W2 rows in two stages of 128
                for (int h = 0; h < 2; ++h) {
                    ok = stage_ready(kInfoMma | 0x400u);
                    if (!ok) return;
                    ptx::tc_fence_after();
                    const uint64_t soff = uint64_t((s * L.stage) >> 4);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        ptx::mma_bf16_ts(tmem + kColO, tmem + kColP + uint32_t((8 * h + k) * 8),
                                         rd_w2 + soff + uint64_t(128 * k), id2, (j | h | k) != 0 ? 1u : 0u);
                    release();
                }
                ptx::mma_commit(B.o_full);
                trace_tile(tr, J, CF_TRB_ML2_DONE);
            };
            if (NJ > 0) ml1(0);
            for (int J = 0; J < NJ && ok; ++J) {
                if (J + 1 < NJ) ml1(J + 1);
                if (ok) ml2(J);
            }
            ptx::mma_commit(B.mma_done);
            volatile uint32_t local_abort = 0;
            ptx::mbar_wait_bounded(B.mma_done, 0, tmo, &local_abort, nullptr, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue groups
        // Group g handles columns [64 g, 64 g + 64) of every chunk; thread = row.
        // A wait that gives up (timeout, or another role's abort) is not left
        // early: every thread still reaches each named barrier in order, on
        // values that no longer matter (the error word is set).
        const int g = (warp - 2) >> 2;
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = q * 32 + lane;
        const int gt = (warp - 2 - 4 * g) * 32 + lane;  // thread within the group
        const bool lead = gt == 0;
        const uint32_t lane_off = uint32_t(q * 32) << 16;
        const uint32_t tS = tmem + lane_off + uint32_t(kCols * g);            // this group's S columns
        const uint32_t tP = tmem + lane_off + kColP + uint32_t(kCols / 2 * g); // and its packed P columns
        const uint32_t tO = tmem + lane_off + kColO + uint32_t(32 * g);       // its O columns (rescale)
        const bool owns_o = 32 * g < kN2;                                     // (N2 = 64: groups 0, 1)
        constexpr int kPrm = OP == 2 ? 2 : 1;  // staged column parameters: b1 (LayerNorm: and gamma1)
        float *const prm = reinterpret_cast<float *>(smem_raw + L.bias) + g * 2 * kPrm * kCols;
        float *const xm = reinterpret_cast<float *>(smem_raw + L.xm);
        float *const stat = reinterpret_cast<float *>(smem_raw + L.stat);
        const float bscale = OP == 0 ? kLog2e : 1.f;
        const float ascale = a.alpha * bscale;  // softmax works in base 2: t = z log2 e
        // the parameters of the group's next chunk, loaded one chunk ahead (threads gt < 64)
        const bool pl = gt < kCols;
        auto ldp = [&](const float *v, int jc) -> float { return (v && pl) ? __ldg(v + jc * kChunk + kCols * g + gt) : 0.f; };
        float nb = ldp(a.b1, 0), ng = 0.f;
        if constexpr (OP == 2) ng = ldp(a.gamma1, 0);
        int J = 0;
        for (int i = 0; i < nrb; ++i) {
            float m = neg_inf(), l = 0.f;  // softmax: running max and sum of this group's columns
            MeanM2 ls{0.f, 0.f};            // LayerNorm: (mean, M2) of this group's columns so far
            float mu0 = 0.f;                // LayerNorm: the row's shift (its first chunk's mean)
            for (int j = 0; j < nc; ++j, ++J) {
                // the chunk's parameters, double-buffered by chunk parity (the previous
                // chunk's barrier ordered every read of this buffer before this write)
                float *const bb = prm + (J & 1) * kPrm * kCols;
                if (pl) {
                    bb[gt] = nb * bscale;
                    if constexpr (OP == 2) bb[kCols + gt] = ng;
                }
                const int jn = j + 1 < nc ? j + 1 : 0;
                nb = ldp(a.b1, jn);
                if constexpr (OP == 2) ng = ldp(a.gamma1, jn);
                ptx::named_bar_sync(1u + uint32_t(g), 128);
                ptx::mbar_wait_bounded(B.s_full, uint32_t(J) & 1u, tmo, abort, a.err, kInfoEpi | uint32_t(g));
                ptx::tc_fence_after();
                if (lead && g < 2) trace_tile(tr, J, g == 0 ? CF_TRB_EPI1_START : CF_TRB_EPI2_START);
                uint32_t x[kFrag][32];  // the chunk's z; then (first halves) its packed bf16 pairs
#pragma unroll
                for (int c = 0; c < kFrag; ++c) ptx::tmem_ld32(tS + c * 32, x[c]);
                ptx::tmem_ld_wait();
                // S is in registers: ML_1 of the next chunk may overwrite it
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B.s_free);
                bool rescale = false;  // softmax: this row raised its reference
                float f = 1.f;
                if constexpr (OP == 0) {
                    // four independent max and sum chains (one long dependent chain
                    // per thread would leave the warp latency-bound)
                    float cmv[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) cmv[r] = neg_inf();
#pragma unroll
                    for (int c = 0; c < kFrag; ++c)
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {  // on packed pairs, three-input max
                            float t0, t1;
                            ptx::fma2(t0, t1, __uint_as_float(x[c][k]), __uint_as_float(x[c][k + 1]), ascale, ascale,
                                      bb[c * 32 + k], bb[c * 32 + k + 1]);
                            x[c][k] = __float_as_uint(t0);
                            x[c][k + 1] = __float_as_uint(t1);
                            cmv[(k >> 1) & 3] = ptx::max3(cmv[(k >> 1) & 3], t0, t1);
                        }
                    // the row's max over the whole chunk: every group's part, through
                    // shared memory
                    float *const xmj = xm + (J & 1) * (128 * kGroups);
                    xmj[g * 128 + row] = fmaxf(fmaxf(cmv[0], cmv[1]), fmaxf(cmv[2], cmv[3]));
                    ptx::named_bar_sync(kGroups + 1, 128 * kGroups);
                    float cm = xmj[row];
#pragma unroll
                    for (int h = 1; h < kGroups; ++h) cm = fmaxf(cm, xmj[h * 128 + row]);
                    // raise the reference only when the chunk's max passes it by 2^8
                    // (always on the row block's first chunk); every group decides alike
                    const bool first = j == 0;
                    const bool raise = first || cm > m + kRescale;
                    const float mn = raise ? fmaxf(m, cm) : m;
                    f = first ? 0.f : ptx::ex2_approx(m - mn);  // 1 when not raised
                    rescale = raise && !first;
                    float sv[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) sv[r] = 0.f;
                    // the chunk's bf16 pairs are packed in place: pair k of fragment c
                    // goes to x[c][k] once x[c][2k] and x[c][2k+1] were read
#pragma unroll
                    for (int c = 0; c < kFrag; ++c)
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float d0, d1;
                            ptx::add2(d0, d1, __uint_as_float(x[c][2 * k]), __uint_as_float(x[c][2 * k + 1]), -mn, -mn);
                            const float e0 = ptx::ex2_approx(d0);
                            const float e1 = ptx::ex2_approx(d1);
                            ptx::add2(sv[(k & 1) * 2], sv[(k & 1) * 2 + 1], sv[(k & 1) * 2], sv[(k & 1) * 2 + 1], e0, e1);
                            x[c][k] = ptx::pack_bf16x2(e0, e1);
                        }
                    l = fmaf(l, f, (sv[0] + sv[1]) + (sv[2] + sv[3]));
                    m = mn;
                    if (lead && g == 0) trace_tile(tr, J, CF_TRB_EPI1_LOCAL);
                } else if constexpr (OP == 2) {
                    // z on packed pairs; (mean, M2) of the chunk's 64 values (two passes
                    // over the registers, four chains), folded into the group's running
                    // pair by counts
                    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < kFrag; ++c)
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            float z0, z1;
                            ptx::fma2(z0, z1, __uint_as_float(x[c][k]), __uint_as_float(x[c][k + 1]), ascale, ascale,
                                      bb[c * 32 + k], bb[c * 32 + k + 1]);
                            x[c][k] = __float_as_uint(z0);
                            x[c][k + 1] = __float_as_uint(z1);
                            ptx::add2(s4[(k >> 1) & 2], s4[((k >> 1) & 2) + 1], s4[(k >> 1) & 2], s4[((k >> 1) & 2) + 1], z0, z1);
                        }
                    const float cmean = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * (1.f / float(kCols));
                    float q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < kFrag; ++c)
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            float d0, d1;
                            ptx::add2(d0, d1, __uint_as_float(x[c][k]), __uint_as_float(x[c][k + 1]), -cmean, -cmean);
                            ptx::fma2(q4[(k >> 1) & 2], q4[((k >> 1) & 2) + 1], d0, d1, d0, d1, q4[(k >> 1) & 2],
                                      q4[((k >> 1) & 2) + 1]);
                        }
                    const MeanM2 cs{cmean, (q4[0] + q4[1]) + (q4[2] + q4[3])};
                    if (j == 0) {
                        // the row's shift: the mean of its first chunk, from every
                        // group's part (every group sums them in the same order)
                        float *const xmi = xm + (i & 1) * (128 * kGroups);
                        xmi[g * 128 + row] = cmean;
                        ptx::named_bar_sync(kGroups + 1, 128 * kGroups);
                        float t = xmi[row];
#pragma unroll
                        for (int h = 1; h < kGroups; ++h) t += xmi[h * 128 + row];
                        mu0 = t * (1.f / float(kGroups));
                        ls = cs;
                    } else {
                        ls = combine_counts(ls, float(kCols * j), cs, float(kCols));
                    }
                    // the shifted, scaled values (z - mu0) gamma1; the statistics and
                    // beta1 are applied to the fp32 output
#pragma unroll
                    for (int c = 0; c < kFrag; ++c)
#pragma unroll
                        for (int k = 0; k < 16; ++k) {  // on packed pairs
                            const int n0 = c * 32 + 2 * k;
                            float d0, d1;
                            ptx::add2(d0, d1, __uint_as_float(x[c][2 * k]), __uint_as_float(x[c][2 * k + 1]), -mu0, -mu0);
                            ptx::mul2(d0, d1, d0, d1, bb[kCols + n0], bb[kCols + n0 + 1]);
                            x[c][k] = ptx::pack_bf16x2(d0, d1);
                        }
                } else {
#pragma unroll
                    for (int c = 0; c < kFrag; ++c)
#pragma unroll
                        for (int k = 0; k < 16; ++k) {  // on packed pairs
                            float x0, x1;
                            ptx::fma2(x0, x1, __uint_as_float(x[c][2 * k]), __uint_as_float(x[c][2 * k + 1]), ascale,
                                      ascale, bb[c * 32 + 2 * k], bb[c * 32 + 2 * k + 1]);
                            gelu_tanh_pair(x0, x1);
                            x[c][k] = ptx::pack_bf16x2(x0, x1);
                        }
                }
                // P and O: ML_2 of the previous chunk is complete (it read P; O holds
                // every earlier chunk)
                if (J > 0)
                    ptx::mbar_wait_bounded(B.o_full, uint32_t(J - 1) & 1u, tmo, abort, a.err, kInfoEpi | 0x10u);
                ptx::tc_fence_after();
                if constexpr (OP == 0) {
                    // O carries the previous chunks against the old reference: rescale
                    // this group's output columns of the rows that raised it
                    // (warp-collective loads and stores: the whole warp takes part)
                    if (owns_o && __any_sync(0xffffffffu, rescale)) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO, o);
                        ptx::tmem_ld_wait();
                        const float fo = rescale ? f : 1.f;
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * fo);
                        ptx::tmem_st32(tO, o);
                    }
                }
#pragma unroll
                for (int c = 0; c < kFrag; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) pk[k] = x[c][k];
                    ptx::tmem_st16(tP + c * 16, pk);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B.p_full);
                if (lead && g == 0) trace_tile(tr, J, CF_TRB_EPI1_DONE);
            }
            // ---------------- the row block's output, once its last ML_2 completed;
            // ML_1 of the next row block's first chunk runs meanwhile
            ptx::mbar_wait_bounded(B.o_full, uint32_t(J - 1) & 1u, tmo, abort, a.err, kInfoEpi | 0x20u);
            ptx::tc_fence_after();
            stream_output<OP, kN2, direct_out<OP, kRes>()>(&a.tmap_o, a.out, a.M, (int(blockIdx.x) + i * int(gridDim.x)) * 128,
                                   tmem + lane_off + kColO, base + L.stg + uint32_t(warp - 2) * 2048u,
                                   stat + (i & 1) * (128 * kGroups) * (OP == 2 ? 2 : 1), l, ls, mu0, a.fold,
                                   float(a.N1), a.eps, g, q, lane, B.mfree, abort,
                                   (lead && g == 0 && tr != nullptr && J - 1 < CF_TRACE_TILES)
                                       ? tr + blockIdx.x * CF_TRACE_SLOTS + 4 + (J - 1) * CF_TRACE_EVENTS +
                                             CF_TRB_EPI2_STORED
                                       : nullptr);
        }
        // every store of this warp has read its staging buffer before the CTA
        // may leave (the writes complete with the grid)
        if (lane == 0) ptx::bulk_wait_group_read0();
        __syncwarp();
    }

    // ------------------------------------------------------------ teardown
    if (threadIdx.x == 64) trace_stamp(tr, 2);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, 512);
    if (threadIdx.x == 64) trace_stamp(tr, 3);
}

// c[0][k] = sum_n gamma1[n] W2[n, k], c[1][k] = sum_n beta1[n] W2[n, k].  Block
// (x, y): columns [64 x, 64 x + 64) (a bf16 pair per lane), rows of split y
// (eight warps, interleaved); the block's sums go to partials[y], and the
// last block of column group x to finish adds the partials in split order
// (a fixed order: the result does not depend on which block finished last).
__global__ void __launch_bounds__(256) b2b_ln_fold_kernel(const uint32_t *__restrict__ w2, const float *__restrict__ gamma,
                                                          const float *__restrict__ beta, float *c, float *part,
                                                          unsigned int *counter, int N1, int N2) {
    // W2, gamma1, beta1 may come from the previous kernel, which may still read
    // c; the stream kernel that follows may start (and read its own inputs)
    // only once every block here has seen the previous grids complete
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    __shared__ float red[8][2][64];
    float(*const red2)[128] = reinterpret_cast<float(*)[128]>(&red[0][0][0]);  // the last block's [2][128]
    __shared__ unsigned int is_last;
    const int x = blockIdx.x, y = blockIdx.y, S = gridDim.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int per = (N1 + S - 1) / S;
    const int n0 = y * per, n1 = min(N1, n0 + per);
    const size_t pitch = size_t(N2 / 2);  // bf16 pairs per row of W2
    const uint32_t *col = w2 + 32 * x + lane;
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll 8
    for (int n = n0 + w; n < n1; n += 8) {
        const uint32_t p = __ldg(col + size_t(n) * pitch);
        const float w0 = __uint_as_float(p << 16), w1 = __uint_as_float(p & 0xffff0000u);
        const float gn = __ldg(gamma + n), bn = __ldg(beta + n);
        g0 = fmaf(gn, w0, g0);
        g1 = fmaf(gn, w1, g1);
        b0 = fmaf(bn, w0, b0);
        b1 = fmaf(bn, w1, b1);
    }
    red[w][0][2 * lane] = g0;
    red[w][0][2 * lane + 1] = g1;
    red[w][1][2 * lane] = b0;
    red[w][1][2 * lane + 1] = b1;
    __syncthreads();
    const int kind = threadIdx.x >> 6, k = threadIdx.x & 63;  // threads < 128
    if (threadIdx.x < 128) {
        float t = 0.f;
#pragma unroll
        for (int h = 0; h < 8; ++h) t += red[h][kind][k];
        part[(size_t(y) * 2 + size_t(kind)) * 128 + size_t(64 * x + k)] = t;
        __threadfence();
    }
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(counter + x, 1u) == unsigned(S - 1) ? 1u : 0u;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // two halves of the splits (S is even), every load issued before the adds
    {
        const int half = threadIdx.x >> 7, v = threadIdx.x & 127, hs = S / 2;
        const float *src = part + (size_t(half * hs) * 2 + size_t(v >> 6)) * 128 + size_t(64 * x + (v & 63));
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < kB2bFoldSplits / 2; ++h)
            if (h < hs) acc[h & 3] += __ldcg(src + size_t(h) * 256);
        red2[half][v] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    __syncthreads();
    if (threadIdx.x < 128) c[kind * N2 + 64 * x + k] = red2[0][threadIdx.x] + red2[1][threadIdx.x];
    if (threadIdx.x == 0) counter[x] = 0u;  // for the next call (every block of this one has counted)
}

template <int OP, bool kRes>
void *stream_fn_n2(int n2) {
    return n2 == 64 ? reinterpret_cast<void *>(&b2b_stream_kernel<OP, 64, kRes>)
                    : reinterpret_cast<void *>(&b2b_stream_kernel<OP, 128, kRes>);
}
void *stream_fn(int op, int n2, bool res) {
    if (op == 0) return res ? stream_fn_n2<0, true>(n2) : stream_fn_n2<0, false>(n2);
    if (op == 2) return res ? stream_fn_n2<2, true>(n2) : stream_fn_n2<2, false>(n2);
    return res ? stream_fn_n2<1, true>(n2) : stream_fn_n2<1, false>(n2);
}

}  // namespace

template <int OP>
Layout layout_for(int K) {
    return K <= kMaxResidentK ? layout<OP, true>() : layout<OP, false>();
}

static Layout layout_op(int op, int K) {
    return op == 0 ? layout_for<0>(K) : op == 2 ? layout_for<2>(K) : layout_for<1>(K);
}

int b2b_stream_stages(int op, int K) { return int(layout_op(op, K).stages); }

int b2b_stream_smem_bytes(int op, int K) { return int(layout_op(op, K).total); }

cudaError_t launch_b2b_ln_fold(const void *W2, const float *gamma1, const float *beta1, int N1, int N2,
                               unsigned char *ws, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(N2 / 64), unsigned(N1 / 64 < kB2bFoldSplits ? (N1 / 64 > 0 ? N1 / 64 : 1)
                                                                              : kB2bFoldSplits));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, b2b_ln_fold_kernel, static_cast<const uint32_t *>(W2), gamma1, beta1,
                              reinterpret_cast<float *>(ws + kB2bFoldOff), reinterpret_cast<float *>(ws + kB2bFoldPartialsOff),
                              reinterpret_cast<unsigned int *>(ws + kB2bFoldCountersOff), N1, N2);
}

cudaError_t launch_b2b_stream(int op, const B2bArgs &a, int ctas, int smem, bool pdl, cudaStream_t stream) {
    if (op < 0 || op > 2) return cudaErrorInvalidValue;
    void *fn = stream_fn(op, a.N2, a.K <= kMaxResidentK);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kThreads);
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

}  // namespace cf
