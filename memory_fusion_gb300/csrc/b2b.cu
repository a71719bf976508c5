// b2b.cu -- back-to-back GEMM with the intermediate kept on chip:
//     O = S . W2,   S = F(alpha * X.W1 + b1) in bf16,   F = row softmax or GELU
// ([ComFuse] B2BGEMM, Eqs. 3-7, Fig. 5).
//
// Design (sm_103a):
//  * A cluster of C CTAs takes one 128-row block; CTA rank r owns the 256
//    columns [256 r, 256 r + 256) of the intermediate P = X.W1 (the output
//    space of MatMul_1 is partitioned along N1, Fig. 5).
//  * ML_1: tcgen05.mma accumulates P_tile (128 x 256, fp32) in tensor memory.
//  * Epi_1: F over P_tile.  For softmax the row statistics (max, sum exp)
//    are reduced over the cluster: every thread sends its row's partial to
//    each CTA with an 8-byte st.async.  S_tile = F(P_tile) is written back to
//    tensor memory as packed bf16 over the consumed columns of P -- S never
//    leaves the SM (Eq. 3: "resident"; here in tensor memory rather than
//    registers, since tcgen05.mma reads its A operand from there).
//  * ML_2: tcgen05.mma with A = S_tile from tensor memory and B = the CTA's
//    256-row slice of W2, streamed through the same operand ring as X and W1
//    (one unified multi-stage buffer for both MatMuls); each CTA accumulates
//    its partial O_tile^(c) = S_tile^(c) W2^(c) (Eq. 4).
//  * Epi_2: the partials are summed over the cluster (Eq. 5) as a
//    reduce-scatter: CTA r owns output columns [r N2/C, (r+1) N2/C); every
//    CTA sends each owner its partial columns with 16-byte st.async, and the
//    owner adds them in rank order (deterministic), rounds to bf16, stores.
//  * The ML_1 of the next row block overlaps Epi_2 (P and O occupy different
//    tensor-memory columns); ML_2 of the next waits until Epi_2 read O.
//  * Every wait is bounded by %globaltimer; a timeout records
//    CF_ERR_DEVICE_TIMEOUT in the workspace error word and the roles drain.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/cf.h"
#include "cf_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"
#include "umma.cuh"

namespace cf {
namespace {

constexpr int kThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
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

__host__ __device__ inline Layout layout(int stages, int C, int N2) {
    Layout L;
    L.ring = 0;
    uint32_t off = uint32_t(stages) * kStageBytes;
    L.slot = off;  // float2 [2 sets][C][128]: softmax partials
    off += 2u * uint32_t(C) * 128u * 8u;
    L.recv = off;  // float [C][128][N2 / C]: the partial output columns this CTA owns
    off += 128u * uint32_t(N2) * 4u;
    L.prm = off;   // float [256]: b1 of this CTA's columns
    off += kN1Slice * 4u;
    L.bars = off;
    off += 256;
    L.total = off;
    return L;
}

struct Bars {
    uint32_t full0, empty0, p_full, s_full, o_full, o_empty, xfull0, rbar, rfree, mma_done, misc;
};
__device__ __forceinline__ Bars bars_at(uint32_t b, int stages) {
    Bars r;
    r.full0 = b;
    r.empty0 = b + 8 * stages;
    r.p_full = b + 16 * stages;
    r.s_full = r.p_full + 8;
    r.o_full = r.s_full + 8;
    r.o_empty = r.o_full + 8;
    r.xfull0 = r.o_empty + 8;  // [2]
    r.rbar = r.xfull0 + 16;
    r.rfree = r.rbar + 8;
    r.mma_done = r.rfree + 8;
    r.misc = r.mma_done + 8;  // u32 tmem base, u32 abort flag
    return r;
}

template <int OP>  // 0 softmax, 1 GELU
__global__ void __launch_bounds__(kThreads, 1) b2b_kernel(const __grid_constant__ B2bArgs a, int stages) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = ptx::smem_u32(smem_raw);
    if ((base & 1023u) != 0u) {
        ptx::griddep_wait();
        if (threadIdx.x == 0) ptx::record_error(a.err, 8u /*CF_ERR_DEVICE_BOUNDS*/, 0x60000000u | (base & 1023u));
        return;
    }
    const int C = a.cluster;
    const int N2 = a.N2;
    const int w = N2 / C;  // output columns owned by each CTA
    const int nk1 = (a.K + kBK - 1) / kBK;  // a ragged last block reads zeros past K
    const int nk2 = kN1Slice / kBK;  // 4
    const Layout L = layout(stages, C, N2);
    const Bars B = bars_at(base + L.bars, stages);
    volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(smem_raw + (B.misc - base));
    volatile uint32_t *abort = misc + 1;
    const uint64_t tmo = a.timeout_ns;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t cid = ptx::cluster_id_x();
    const uint32_t ncl = ptx::nclusters_x();
    const int RB = (a.M + 127) / 128;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(B.full0 + 8 * s, 1);
            ptx::mbar_init(B.empty0 + 8 * s, 1);
        }
        ptx::mbar_init(B.p_full, 1);
        ptx::mbar_init(B.s_full, 4);
        ptx::mbar_init(B.o_full, 1);
        ptx::mbar_init(B.o_empty, 4);
        ptx::mbar_init(B.xfull0, 1);
        ptx::mbar_init(B.xfull0 + 8, 1);
        ptx::mbar_init(B.rbar, 1);
        ptx::mbar_init(B.rfree, 4u * uint32_t(C));
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
    const uint32_t tmem = misc[0];
    const uint32_t tP = tmem;                 // P, then S (bf16 pairs) over its first 128 columns
    const uint32_t tO = tmem + kN1Slice;      // O partial, N2 columns
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_last();
            uint32_t s = 0, ph = 0, it = 0;
            bool ok = true;
            const uint32_t w2_tx = uint32_t(kBK) * uint32_t(N2) * 2u;
            for (int rb = int(cid); rb < RB && ok; rb += int(ncl)) {
                const int m0 = rb * 128;
                for (int kb = 0; kb < nk1 + nk2; ++kb) {
                    ok = ptx::mbar_wait_bounded(B.empty0 + 8 * s, ph ^ 1u, tmo, abort, a.err, kInfoProducer | s);
                    if (!ok) break;
                    const uint32_t sa = base + L.ring + s * kStageBytes;
                    const uint32_t fb = B.full0 + 8 * s;
                    if (kb < nk1) {  // MatMul_1: X and this CTA's W1 columns
                        ptx::mbar_arrive_expect_tx(fb, uint32_t(kStageBytes));
                        ptx::tma_load_2d(sa, &a.tmap_x, fb, kb * kBK, m0);
                        ptx::tma_load_3d_hint(sa + kABytes, &a.tmap_w1, fb, 0, kb * kBK, int(rank) * (kN1Slice / 64),
                                              pol_w);
                    } else {  // MatMul_2: 64 rows of this CTA's W2 slice
                        ptx::mbar_arrive_expect_tx(fb, w2_tx);
                        ptx::tma_load_3d_hint(sa + kABytes, &a.tmap_w2, fb, 0,
                                              int(rank) * kN1Slice + (kb - nk1) * kBK, 0, pol_w);
                    }
                    ++it;
                    if (++s == uint32_t(stages)) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
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
            const uint32_t id2 = idesc_bf16(128, N2);  // A from tensor memory (K-major), B = W2 MN-major
            const uint64_t ad0 = sw128_desc(base + L.ring, 16, 1024);
            const uint64_t bd0 = sw128_desc(base + L.ring + kABytes, 8192, 1024);
            uint32_t s = 0, ph = 0;
            int tile = 0;
            bool ok = true;
            for (int rb = int(cid); rb < RB && ok; rb += int(ncl), ++tile) {
                const uint32_t tph = uint32_t(tile) & 1u;
                // ML_1 (P's columns are free: ML_2 of the previous tile, issued
                // earlier on this thread, has read S out of them)
                for (int kb = 0; kb < nk1; ++kb) {
                    if (!ptx::mbar_try_wait(B.full0 + 8 * s, ph)) {
                        ok = ptx::mbar_wait_bounded(B.full0 + 8 * s, ph, tmo, abort, a.err, kInfoMma | s);
                        if (!ok) break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t soff = uint64_t((s * uint32_t(kStageBytes)) >> 4);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        ptx::mma_bf16(tP, ad0 + soff + uint64_t(2 * k), bd0 + soff + uint64_t(128 * k), id1,
                                      (kb | k) != 0 ? 1u : 0u);
                    ptx::mma_commit(B.empty0 + 8 * s);
                    if (++s == uint32_t(stages)) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(B.p_full);
                // S is in tensor memory, and Epi_2 of the previous tile read O
                ok = ptx::mbar_wait_bounded(B.s_full, tph, tmo, abort, a.err, kInfoMma | 0x100u);
                if (!ok) break;
                ok = ptx::mbar_wait_bounded(B.o_empty, tph ^ 1u, tmo, abort, a.err, kInfoMma | 0x200u);
                if (!ok) break;
                ptx::tc_fence_after();
                // ML_2: O^(c) = S^(c) W2^(c), K = 256 in four 64-deep stages; per
                // MMA, K = 16 bf16 of A = 8 tensor-memory columns
                for (int kb = 0; kb < nk2; ++kb) {
                    if (!ptx::mbar_try_wait(B.full0 + 8 * s, ph)) {
                        ok = ptx::mbar_wait_bounded(B.full0 + 8 * s, ph, tmo, abort, a.err, kInfoMma | 0x300u | s);
                        if (!ok) break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t soff = uint64_t((s * uint32_t(kStageBytes)) >> 4);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        ptx::mma_bf16_ts(tO, tP + uint32_t(kb * 32 + k * 8), bd0 + soff + uint64_t(128 * k), id2,
                                         (kb | k) != 0 ? 1u : 0u);
                    ptx::mma_commit(B.empty0 + 8 * s);
                    if (++s == uint32_t(stages)) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(B.o_full);
            }
            ptx::mma_commit(B.mma_done);
            volatile uint32_t local_abort = 0;
            ptx::mbar_wait_bounded(B.mma_done, 0, tmo, &local_abort, nullptr, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quadrant
        const int row = q * 32 + lane;
        const bool lead = (warp == 2 && lane == 0);
        const uint32_t tq = uint32_t(q * 32) << 16;
        float *const prm = reinterpret_cast<float *>(smem_raw + L.prm);
        const float2 *slot = reinterpret_cast<const float2 *>(smem_raw + L.slot);
        const float *recv = reinterpret_cast<const float *>(smem_raw + L.recv);
        const int n0 = int(rank) * kN1Slice;
        for (int c = (warp - 2) * 32 + lane; c < kN1Slice; c += 128) prm[c] = a.b1 ? __ldg(a.b1 + n0 + c) : 0.f;
        ptx::named_bar_sync(1, 128);
        int tile = 0;
        for (int rb = int(cid); rb < RB; rb += int(ncl), ++tile) {
            const uint32_t tph = uint32_t(tile) & 1u;
            const int m0 = rb * 128;
            if (!ptx::mbar_wait_bounded(B.p_full, tph, tmo, abort, a.err, kInfoEpi)) break;
            ptx::tc_fence_after();
            // ---------------- Epi_1: S = F(alpha * P + b1), bf16 into tensor memory
            if constexpr (OP == 0) {
                float m = neg_inf(), ssum = 0.f, mrun[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tP + tq + c * 32, v);
                    ptx::tmem_ld_wait();
                    float z[32], cm = neg_inf();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        z[j] = fmaf(a.alpha, __uint_as_float(v[j]), prm[c * 32 + j]);
                        cm = fmaxf(cm, z[j]);
                    }
                    const float mn = fmaxf(m, cm);
                    float s = ssum * ptx::ex2_approx((m - mn) * kLog2e);
                    const float off = mn * kLog2e;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float e = ptx::ex2_approx(fmaf(z[j], kLog2e, -off));
                        s += e;
                        v[j] = __float_as_uint(e);
                    }
                    ssum = s;
                    m = mn;
                    mrun[c] = mn;
                    ptx::tmem_st32(tP + tq + c * 32, v);
                }
                ptx::tmem_st_wait();
                // row statistics over the cluster: every thread sends its row's
                // (max, sum) to each CTA; the gatherers fold them in rank order
                const uint32_t xs = uint32_t(tile) & 1u, xph = (uint32_t(tile) >> 1) & 1u;
                const uint32_t xb = B.xfull0 + 8 * xs;
                float2 st = make_float2(m, ssum);
                if (C > 1 && !*abort) {
                    if (lead) ptx::mbar_arrive_expect_tx(xb, uint32_t(C) * 1024u);
                    const uint32_t mine = base + L.slot + (xs * uint32_t(C) + rank) * 1024u + uint32_t(row) * 8u;
                    for (int r = 0; r < C; ++r)
                        ptx::st_async_f2(ptx::mapa(mine, uint32_t(r)), m, ssum, ptx::mapa(xb, uint32_t(r)));
                    ptx::mbar_wait_bounded<true>(xb, xph, tmo, abort, a.err, kInfoEpi | 0x10u | xs);
                    const float2 *sr = slot + size_t(xs) * size_t(C) * 128u + row;
                    st = sr[0];
                    for (int r = 1; r < C; ++r) {
                        const MaxSum mm = combine_maxsum(MaxSum{st.x, st.y}, MaxSum{sr[r * 128].x, sr[r * 128].y});
                        st = make_float2(mm.m, mm.s);
                    }
                }
                const float inv = 1.0f / st.y;
                // S = exp(z - m_row) / s_row, packed bf16 over the consumed P columns
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32], sv[16];
                    ptx::tmem_ld32(tP + tq + c * 32, v);
                    ptx::tmem_ld_wait();
                    const float f = ptx::ex2_approx((mrun[c] - st.x) * kLog2e) * inv;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        sv[j] = ptx::pack_bf16x2(__uint_as_float(v[2 * j]) * f, __uint_as_float(v[2 * j + 1]) * f);
                    ptx::tmem_st16(tP + tq + c * 16, sv);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32], sv[16];
                    ptx::tmem_ld32(tP + tq + c * 32, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float x0 = gelu_tanh_dev(fmaf(a.alpha, __uint_as_float(v[2 * j]), prm[c * 32 + 2 * j]));
                        const float x1 =
                            gelu_tanh_dev(fmaf(a.alpha, __uint_as_float(v[2 * j + 1]), prm[c * 32 + 2 * j + 1]));
                        sv[j] = ptx::pack_bf16x2(x0, x1);
                    }
                    ptx::tmem_st16(tP + tq + c * 16, sv);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(B.s_full);
            // ---------------- Epi_2: reduce-scatter of the partial outputs over the cluster
            if (!ptx::mbar_wait_bounded(B.o_full, tph, tmo, abort, a.err, kInfoEpi | 0x20u)) break;
            ptx::tc_fence_after();
            if (lead) ptx::mbar_arrive_expect_tx(B.rbar, 128u * uint32_t(N2) * 4u);
            // every owner has read the previous tile's partials out of its buffer
            if (tile > 0 &&
                !ptx::mbar_wait_bounded<true>(B.rfree, (tph ^ 1u), tmo, abort, a.err, kInfoEpi | 0x28u))
                break;
            for (int c = 0; c < N2 / 32; ++c) {
                uint32_t v[32];
                ptx::tmem_ld32(tO + tq + c * 32, v);
                ptx::tmem_ld_wait();
                if (*abort) continue;
                // columns [32c, 32c+32) go to their owners, w columns each
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const int col = c * 32 + j;
                    const int owner = col / w, k = col % w;
                    const uint32_t dst =
                        base + L.recv + ((rank * 128u + uint32_t(row)) * uint32_t(w) + uint32_t(k)) * 4u;
                    ptx::st_async_f4(ptx::mapa(dst, uint32_t(owner)), __uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                     __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]),
                                     ptx::mapa(B.rbar, uint32_t(owner)));
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(B.o_empty);  // ML_2 of the next tile may overwrite O
            if (!ptx::mbar_wait_bounded<true>(B.rbar, tph, tmo, abort, a.err, kInfoEpi | 0x30u)) break;
            // O[row, rank*w .. +w) = sum over the cluster, in rank order
            if (m0 + row < a.M) {
                uint16_t *orow = a.out + size_t(m0 + row) * size_t(N2) + size_t(rank) * size_t(w);
                for (int k0 = 0; k0 < w; k0 += 8) {
                    float acc[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[k] = recv[(0 * 128 + row) * w + k0 + k];
                    for (int r = 1; r < C; ++r)
#pragma unroll
                        for (int k = 0; k < 8; ++k) acc[k] += recv[(r * 128 + row) * w + k0 + k];
                    uint4 o;
                    o.x = ptx::pack_bf16x2(acc[0], acc[1]);
                    o.y = ptx::pack_bf16x2(acc[2], acc[3]);
                    o.z = ptx::pack_bf16x2(acc[4], acc[5]);
                    o.w = ptx::pack_bf16x2(acc[6], acc[7]);
                    *reinterpret_cast<uint4 *>(orow + k0) = o;
                }
            }
            // this warp's rows of the buffer are free again: one arrival at every sender
            __syncwarp();
            if (lane == 0)
                for (int r = 0; r < C; ++r) ptx::mbar_arrive_cluster(ptx::mapa(B.rfree, uint32_t(r)));
        }
    }

    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_sync();  // no CTA leaves while a peer may still write its shared memory
    if (warp == 1) ptx::tmem_dealloc(tmem, 512);
}

template <int OP>
void *b2b_fn() {
    return reinterpret_cast<void *>(&b2b_kernel<OP>);
}

}  // namespace

int b2b_smem_bytes(int stages, int cluster, int n2) { return int(layout(stages, cluster, n2).total); }

int b2b_max_active_clusters(int op, int cluster, int smem) {
    void *fn = op == 0 ? b2b_fn<0>() : b2b_fn<1>();
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
    void *fn = op == 0 ? b2b_fn<0>() : b2b_fn<1>();
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
