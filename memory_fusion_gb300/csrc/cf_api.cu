// cf_api.cu -- the C ABI of libcf (declared in include/cf.h): argument and
// alignment checks, the launch planner (row-to-CTA/cluster mapping, residency
// check for the in-kernel barrier), TMA descriptor construction, launches,
// and the device error word.  No allocation happens on any call path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/cf.h"
#include "cf_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

cf_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = int(e);
    return CF_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

constexpr int kMaxSmem = 232448;  // 227 KB dynamic shared memory per CTA (sm_100 family)
constexpr uint32_t kDefaultTimeoutUs = 200000;

std::mutex g_mu;

// -------------------------------------------------------------------------
// driver entry point for tensor-map encoding (no link-time libcuda dependency)
// -------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box (box_cols x box_rows);
// out-of-range elements read as zero and are not written.
bool make_tmap_bf16(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                    uint32_t box_rows, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// W [K, N] bf16 row-major as a 3-D tensor {64 columns, K rows, N/64 column
// blocks} with strides N*2 and 128 bytes; a box of `blocks` 64x64 blocks lands
// as consecutive 8 KB, 128B-swizzled blocks (the MN-major B operand layout)
bool make_tmap_w(CUtensorMap *m, const void *ptr, uint64_t K, uint64_t N, uint32_t blocks, uint32_t rows = 64) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, K, N / 64};
    cuuint64_t strides[2] = {N * 2, 128};
    cuuint32_t box[3] = {64, rows, blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// W column blocks one CTA stages per k-block (a CTA of a pair: half the tile's)
uint32_t w_blocks(int n_slice, int cluster_m) { return uint32_t(n_slice / 64 / (cluster_m == 2 ? 2 : 1)); }

// 2-D fp32 tensor map over a row-major [rows, cols] matrix for TMA stores of
// 16-column x 32-row blocks (64-byte rows, 64B swizzle)
bool make_tmap_f32_store(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D fp32 tensor map over a row-major [rows, cols] matrix, box (box_cols x
// box_rows), no swizzle: loads read zeros outside, stores are clipped
bool make_tmap_f32(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                   uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// -------------------------------------------------------------------------
// occupancy cache: max co-resident clusters for (device, kind, cluster, smem)
// -------------------------------------------------------------------------
int max_active_cached(int device, int kind, bool pair, int cluster, int smem) {
    static std::map<std::tuple<int, int, int, int, int>, int> cache;
    auto key = std::make_tuple(device, kind, pair ? 1 : 0, cluster, smem);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = cf::gemm_fused_max_active_clusters(kind, pair, cluster, smem);
    std::lock_guard<std::mutex> lk(g_mu);
    cache[key] = n;
    return n;
}

int gemm_stages_for(int n_slice, int cluster, int requested, bool pair, bool leader, int stg_bufs = 1) {
    int s = requested > 0 ? requested : 6;
    while (s > 2 && cf::gemm_fused_smem_bytes(s, cluster, n_slice, pair, leader, stg_bufs) > kMaxSmem) --s;
    return s;
}

}  // namespace

namespace cf {

bool current_device_info(DeviceInfo *out) {
    static std::map<int, DeviceInfo> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(dev);
        if (it != cache.end()) {
            *out = it->second;
            return true;
        }
    }
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    cache[dev] = d;
    *out = d;
    return true;
}

}  // namespace cf

// =========================================================================
// C ABI
// =========================================================================
extern "C" {

const char *cf_status_string(cf_status s) {
    switch (s) {
        case CF_OK: return "CF_OK";
        case CF_ERR_INVALID_ARG: return "CF_ERR_INVALID_ARG";
        case CF_ERR_UNSUPPORTED: return "CF_ERR_UNSUPPORTED";
        case CF_ERR_MISALIGNED: return "CF_ERR_MISALIGNED";
        case CF_ERR_WORKSPACE_TOO_SMALL: return "CF_ERR_WORKSPACE_TOO_SMALL";
        case CF_ERR_NOT_RESIDENT: return "CF_ERR_NOT_RESIDENT";
        case CF_ERR_CUDA: return "CF_ERR_CUDA";
        case CF_ERR_DEVICE_TIMEOUT: return "CF_ERR_DEVICE_TIMEOUT";
        case CF_ERR_DEVICE_BOUNDS: return "CF_ERR_DEVICE_BOUNDS";
        case CF_ERR_NO_DEVICE: return "CF_ERR_NO_DEVICE";
        default: return "CF_ERR_UNKNOWN";
    }
}

int cf_version(void) { return 100; }

int cf_last_cuda_error(void) { return g_last_cuda_error; }

void cf_tuning_default(cf_tuning *t) {
    if (t) std::memset(t, 0, sizeof(*t));
}

cf_status cf_plan_gemm_fused(int64_t M, int64_t N, int64_t K, int32_t sm_count,
                             const int32_t max_active_clusters[17], const cf_tuning *tuning, cf_plan *plan) {
    if (!plan || !max_active_clusters || M < 0 || N <= 0 || K <= 0 || sm_count <= 0) return CF_ERR_INVALID_ARG;
    cf_tuning tz;
    cf_tuning_default(&tz);
    const cf_tuning &t = tuning ? *tuning : tz;
    if (K % 64 != 0 || N % 64 != 0) return CF_ERR_UNSUPPORTED;
    if (M > (int64_t(1) << 31) - 128 || N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return CF_ERR_UNSUPPORTED;
    // n_slice candidates: the requested one, else the widest of 256/128/64 that
    // divides N and, when 512 divides N, the wide tile (512 columns: all of
    // tensor memory, both epilogue groups on one tile)
    const int ns_narrow = (N % 256 == 0) ? 256 : (N % 128 == 0) ? 128 : 64;
    if (t.n_slice != 0 && ((t.n_slice != 64 && t.n_slice != 128 && t.n_slice != 256 && t.n_slice != 512) ||
                           N % t.n_slice != 0))
        return CF_ERR_UNSUPPORTED;
    if (N / ns_narrow > 16 * 64) return CF_ERR_UNSUPPORTED;
    const int rb = int((M + cf::kBlockM - 1) / cf::kBlockM);
    const int nk = int(K / 64);
    // Choose n_slice, C_N (CTAs along a row, a divisor of the CTAs per row) and
    // C_M (row blocks per cluster: 2 = CTA pairs sharing one cta_group::2 MMA
    // stream) by predicted time.  The persistent grid holds ncl clusters (never
    // more than can be resident); each takes per = ceil(T / ncl) of T =
    // ceil(row_blocks / C_M) * G tickets, one tile per CTA each.  With two TMEM
    // accumulators and two epilogue groups, tiles go in rounds of two: a round
    // costs max(2 mainloops, one epilogue).  A wide tile has one accumulator, so
    // its tiles run one after another: mainloop + epilogue each.  Constants
    // measured on GB300 with the device trace (128x256 tiles per CTA):
    //   mainloop  ~ 0.35 us per 64-deep k-block for a CTA pair, 0.50 us single
    //               (per 256 columns of W staged)
    //   epilogue  ~ 1.4 us + 3.1 us per 256 columns a thread's row slice holds
    //               (4.5 us for a 256-column slice); + 1.5 + 0.2 G us when
    //               the row spans G > 1 clusters
    //               (the global barrier waits for the slowest of G clusters);
    //               + 0.5 us for a CTA pair when K < 512
    //               + 0.05 C_N us for the cluster exchange (peer all-to-all), or
    //               1 us when it goes through a leader (two hops)
    //   skew      ~ 0.05 G us per tile when G > 1
    // Rows wider than one row group need all G clusters of a row block
    // resident (ncl >= G); a wide tile's row never leaves its cluster (G = 1).
    auto predict = [&](int ns, int cn, int cm, int *ncl_out) -> double {
        const int cpr = int(N / ns);
        const int c = cn * cm;
        const bool wide = ns > 256;
        if (cn < 1 || c > 16 || cpr % cn != 0 || max_active_clusters[c] <= 0) return -1.0;
        if (cm == 2 && (ns < 128 || rb < 2 || wide)) return -1.0;
        const int g = cpr / cn;
        if (wide && (g > 1 || cn > 8)) return -1.0;  // a wide row: one cluster of <= 8 (<= 16 partials)
        int n = max_active_clusters[c];
        if (t.max_clusters > 0) n = std::min(n, int(t.max_clusters));
        if (g > 1 && n < g) return -1.0;
        // With fewer resident clusters than two row groups, every row group's G
        // tickets straddle two rounds of the static ticket order (its first
        // clusters wait at the global barrier for a whole mainloop) and every
        // cluster's column group changes from ticket to ticket, so each row
        // block streams all of W again through L2.  Exactly G clusters keep one
        // column group each: the rounds align with the row groups and each W
        // column block is read once per launch (wide LN 8192x16384x2048: DRAM
        // reads 282 -> 110 MB a launch, 413 -> 406 us under the power cap,
        // 391 -> 398 us in a short burst).
        if (g > 1 && n < 2 * g) n = g;
        const int64_t T = int64_t((rb + cm - 1) / cm) * g;
        if (T < n) n = int(T);
        const int64_t per = (T + n - 1) / n;
        const double t_main = nk * (cm == 2 ? 0.35 : 0.50) * (ns / 256.0);
        const int pm = t.peer_max == 0 ? 8 : t.peer_max;
        const double t_x = (pm < 0 || cn > pm) ? 1.0 : 0.05 * cn;
        const double cols = wide ? 256.0 : double(ns);  // a wide tile splits its columns over both groups
        const double t_epi = 1.4 + 3.1 * (cols / 256.0) + t_x + (g > 1 ? 1.5 + 0.2 * g : 0.0) +
                             (cm == 2 && nk < 8 ? 0.5 : 0.0);
        *ncl_out = n;
        if (wide) return double(per) * (t_main + t_epi);
        return double((per + 1) / 2) * std::max(2.0 * t_main, t_epi) + t_main + (g > 1 ? per * 0.05 * g : 0.0);
    };
    int ns = 0, C = 0, CMs = 0, ncl = 0;
    {
        double best = 0.0;
        // narrower tiles than the widest that divides N only when the widest
        // cannot give every SM a tile: more CTAs per row then shorten the
        // latency chain (a one-row-block LayerNorm: 10.3 us at 256 columns,
        // 6.8 us at 64 columns over a cluster of 8)
        const bool few = int64_t(rb) * (N / ns_narrow) < int64_t(sm_count);
        const int cand[4] = {t.n_slice != 0 ? int(t.n_slice) : ns_narrow,
                             (t.n_slice == 0 && N % 512 == 0) ? 512 : 0,
                             (t.n_slice == 0 && few && ns_narrow > 128) ? 128 : 0,
                             (t.n_slice == 0 && few && ns_narrow > 64) ? 64 : 0};
        for (int ci = 0; ci < 4; ++ci) {
            const int nsc = cand[ci];
            if (nsc == 0) continue;
            const int cpr = int(N / nsc);
            for (int cm = 2; cm >= 1; --cm) {
                if (t.cluster_m > 0 && cm != t.cluster_m) continue;
                for (int cn = std::min(16, cpr); cn >= 1; --cn) {  // larger clusters win ties
                    if (t.cluster_size > 0 && cn != t.cluster_size) continue;
                    int n = 0;
                    const double e = predict(nsc, cn, cm, &n);
                    if (e > 0.0 && (C == 0 || e < best * (1.0 - 1e-9))) {
                        best = e;
                        ns = nsc;
                        C = cn;
                        CMs = cm;
                        ncl = n;
                    }
                }
            }
        }
        if (C == 0) {
            const int cpr = int(N / cand[0]);
            if (t.cluster_size > 16 || (t.cluster_size > 0 && cpr % t.cluster_size != 0)) return CF_ERR_UNSUPPORTED;
            if (t.cluster_m > 2 || t.cluster_m < 0) return CF_ERR_UNSUPPORTED;
            // a wide tile's row must fit one cluster of at most 8, without pairs
            if (cand[0] > 256 && (cpr > 8 || t.cluster_m == 2 || (t.cluster_size > 0 && t.cluster_size != cpr)))
                return CF_ERR_UNSUPPORTED;
            return CF_ERR_NOT_RESIDENT;
        }
    }
    const int cpr = int(N / ns);
    const int G = cpr / C;
    const int peer_max = t.peer_max == 0 ? 8 : t.peer_max;
    plan->n_slice = ns;
    plan->ctas_per_row = cpr;
    plan->cluster_size = C;
    plan->groups = G;
    plan->leader_mode = (peer_max < 0 || C > peer_max) ? 1 : 0;
    plan->row_blocks = rb;
    plan->clusters = std::max(ncl, 1);
    {
        // operand ring first; a second output staging buffer per warp only where
        // it costs no ring stage the K loop can use (at most nk + 1 are useful)
        const bool pair = CMs == 2, lead = plan->leader_mode != 0;
        int st = gemm_stages_for(ns, C, t.stages, pair, lead, 1);
        int sb = 1;
        const int useful = std::max(2, nk + 1);
        if (t.stages <= 0 && st > useful) st = useful;
        if (cf::gemm_fused_smem_bytes(st, C, ns, pair, lead, 2) <= kMaxSmem) sb = 2;
        plan->stages = st;
        plan->staging_buffers = sb;
        plan->smem_bytes = cf::gemm_fused_smem_bytes(st, C, ns, pair, lead, sb);
    }
    plan->cluster_m = CMs;
    if (plan->smem_bytes > kMaxSmem) return CF_ERR_UNSUPPORTED;
    return CF_OK;
}

size_t cf_gemm_fused_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)K;
    if (M < 0 || N <= 0) return cf::kErrBytes;
    size_t rb = size_t((M + cf::kBlockM - 1) / cf::kBlockM);
    rb += rb & 1;  // row blocks are padded to whole clusters of two
    const size_t gmax = size_t((N + 63) / 64) + 1;  // cluster groups, rounded up to even
    return cf::kErrBytes + cf::align_up(8 * rb, 256) + rb * gmax * 128 * sizeof(float2);
}

size_t cf_stitch_workspace_size(int64_t rows, int64_t cols) {
    (void)rows;
    (void)cols;
    return cf::kErrBytes;
}

cf_status cf_workspace_init(void *ws, size_t bytes, cf_stream_t stream) {
    if (!ws) return CF_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(ws, 0, bytes, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CF_OK : cuda_fail(e);
}

cf_status cf_get_device_status(void *ws, cf_stream_t stream, int32_t *info) {
    if (!ws) return CF_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t w[2] = {0, 0};
    e = cudaMemcpy(w, ws, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (info) *info = int32_t(w[1]);
    if (w[0] != 0) {
        e = cudaMemset(ws, 0, sizeof(w));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return cf_status(w[0]);
}

// -------------------------------------------------------------------------
// stitched subgraph
// -------------------------------------------------------------------------
// Row-task mapping of the stitched row subgraphs ([AStitch] "Adaptive thread
// mapping"): rows of at most 32 float4 groups are packed several to a warp
// (lanes per row = groups rounded up to a power of two); wider rows are split
// over a cluster of C CTAs, C from the row count and the SM count.
static cf_status plan_row_mapping(int64_t rows, int64_t cols, const cf_tuning &t, const cf::DeviceInfo &dev,
                                  cf::StitchPlan *pp, int (*packed_bps)(int, bool), int ctas_per_sm = 1) {
    cf::StitchPlan &p = *pp;
    p.pdl = t.disable_pdl == 0;
    p.timeout_ns = 1000ull * (t.timeout_us ? t.timeout_us : kDefaultTimeoutUs);
    const int ng = int((cols + 3) / 4);
    int mapping = t.stitch_mapping;
    if (mapping == 0) mapping = (ng <= 32) ? 1 : 2;
    if (mapping == 1 && ng > 32) return CF_ERR_UNSUPPORTED;
    p.mapping = mapping;
    if (mapping == 1) {
        p.lpr = next_pow2(ng);
        const int rows_per_cta_iter = 8 * (32 / p.lpr) * cf::kPackedUnroll;
        const int64_t want = (rows + rows_per_cta_iter - 1) / rows_per_cta_iter;
        int bps = packed_bps(p.lpr, p.vec);
        if (bps <= 0) bps = 1;
        p.grid = int(std::min<int64_t>(want, int64_t(dev.sm_count) * bps));
    } else if (mapping == 2) {
        int C = t.cluster_size;
        if (C <= 0) {
            const int c_min = (ng + 256 * 16 - 1) / (256 * 16);
            // about ctas_per_sm CTAs per SM for few rows (measured on the 64x30000
            // shape: the softmax and add + LayerNorm are fastest at 8 CTAs per row,
            // two or more per SM, so an SM's loads are spread over several CTAs'
            // exchanges; 16 lost to the cluster barriers)
            int c_par = 1;
            const int64_t want = int64_t(dev.sm_count) * ctas_per_sm;
            if (rows < want) c_par = next_pow2(int((want + rows - 1) / rows));
            C = std::max(c_min, c_par);
            C = std::min(C, 16);
            while (C > 1 && C > ng) C >>= 1;
        }
        if (C < 1 || C > 16) return CF_ERR_UNSUPPORTED;
        const int gpc = (ng + C - 1) / C;
        const int v = next_pow2((gpc + 255) / 256);
        if (v > 16) return CF_ERR_UNSUPPORTED;
        p.cluster = C;
        p.per_thread = v;
        const int peer_max = t.peer_max == 0 ? 8 : t.peer_max;
        p.leader = (peer_max < 0 || C > peer_max) ? 1 : 0;
        int64_t clusters = std::min<int64_t>(rows, 8192);
        if (t.max_clusters > 0) clusters = std::min<int64_t>(clusters, t.max_clusters);
        p.grid = int(clusters * C);
    } else {
        return CF_ERR_INVALID_ARG;
    }
    return CF_OK;
}

cf_status cf_stitch_rowreduce_broadcast_ex(const float *A, const float *row_bias, float *out, int64_t rows,
                                           int64_t cols, void *ws, size_t ws_bytes, cf_stream_t stream,
                                           const cf_tuning *tuning) {
    if (rows < 0 || cols < 0) return CF_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CF_OK;
    if (!A || !row_bias || !out || !ws) return CF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(row_bias)) & 3u)
        return CF_ERR_MISALIGNED;
    if (cols > 262144) return CF_ERR_UNSUPPORTED;
    if (ws_bytes < cf_stitch_workspace_size(rows, cols)) return CF_ERR_WORKSPACE_TOO_SMALL;
    cf_tuning tz;
    cf_tuning_default(&tz);
    const cf_tuning &t = tuning ? *tuning : tz;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;

    cf::StitchPlan p;
    p.vec = (cols % 4 == 0) && aligned16(A) && aligned16(out);
    cf_status st = plan_row_mapping(rows, cols, t, dev, &p, cf::stitch_packed_blocks_per_sm, 2);
    if (st != CF_OK) return st;
    cudaError_t e = cf::launch_stitch(p, A, row_bias, out, rows, cols, static_cast<uint32_t *>(ws),
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return CF_OK;
}


cf_status cf_stitch_powadd_softmax_ex(const float *A, const float *w, float p, float *out, int64_t rows,
                                      int64_t cols, void *ws, size_t ws_bytes, cf_stream_t stream,
                                      const cf_tuning *tuning) {
    if (rows < 0 || cols < 0) return CF_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CF_OK;
    if (!A || !w || !out || !ws) return CF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(w)) & 3u)
        return CF_ERR_MISALIGNED;
    if (cols > 262144) return CF_ERR_UNSUPPORTED;
    if (ws_bytes < cf_stitch_workspace_size(rows, cols)) return CF_ERR_WORKSPACE_TOO_SMALL;
    cf_tuning tz;
    cf_tuning_default(&tz);
    const cf_tuning &t = tuning ? *tuning : tz;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;

    cf::StitchPlan pl;
    pl.vec = (cols % 4 == 0) && aligned16(A) && aligned16(out);
    cf_status st = plan_row_mapping(rows, cols, t, dev, &pl, cf::stitch_packed_blocks_per_sm, 2);
    if (st != CF_OK) return st;
    cudaError_t e = cf::launch_stitch(pl, A, nullptr, out, rows, cols, static_cast<uint32_t *>(ws),
                                      reinterpret_cast<cudaStream_t>(stream), w, p);
    if (e != cudaSuccess) return cuda_fail(e);
    return CF_OK;
}

cf_status cf_stitch_powadd_softmax(const float *A, const float *w, float p, float *out, int64_t rows, int64_t cols,
                                   void *ws, size_t ws_bytes, cf_stream_t stream) {
    return cf_stitch_powadd_softmax_ex(A, w, p, out, rows, cols, ws, ws_bytes, stream, nullptr);
}

cf_status cf_stitch_rowreduce_broadcast(const float *A, const float *row_bias, float *out, int64_t rows,
                                        int64_t cols, void *ws, size_t ws_bytes, cf_stream_t stream) {
    return cf_stitch_rowreduce_broadcast_ex(A, row_bias, out, rows, cols, ws, ws_bytes, stream, nullptr);
}

cf_status cf_stitch_add_layernorm_ex(const float *A, const float *R, const float *gamma, const float *beta,
                                     float *out, int64_t rows, int64_t cols, float eps, void *ws, size_t ws_bytes,
                                     cf_stream_t stream, const cf_tuning *tuning) {
    if (rows < 0 || cols < 0) return CF_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CF_OK;
    if (!A || !gamma || !beta || !out || !ws) return CF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(R) | reinterpret_cast<uintptr_t>(out) |
         reinterpret_cast<uintptr_t>(gamma) | reinterpret_cast<uintptr_t>(beta)) & 3u)
        return CF_ERR_MISALIGNED;
    if (cols > 262144) return CF_ERR_UNSUPPORTED;
    if (ws_bytes < cf_stitch_workspace_size(rows, cols)) return CF_ERR_WORKSPACE_TOO_SMALL;
    cf_tuning tz;
    cf_tuning_default(&tz);
    const cf_tuning &t = tuning ? *tuning : tz;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;
    cf::StitchPlan p;
    p.vec = (cols % 4 == 0) && aligned16(A) && aligned16(out) && (R == nullptr || aligned16(R)) &&
            aligned16(gamma) && aligned16(beta);
    cf_status st = plan_row_mapping(rows, cols, t, dev, &p, cf::addln_packed_blocks_per_sm, 2);
    if (st != CF_OK) return st;
    cudaError_t e = cf::launch_add_layernorm(p, A, R, gamma, beta, out, rows, cols, eps,
                                             static_cast<uint32_t *>(ws), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return CF_OK;
}

cf_status cf_stitch_add_layernorm(const float *A, const float *R, const float *gamma, const float *beta,
                                  float *out, int64_t rows, int64_t cols, float eps, void *ws, size_t ws_bytes,
                                  cf_stream_t stream) {
    return cf_stitch_add_layernorm_ex(A, R, gamma, beta, out, rows, cols, eps, ws, ws_bytes, stream, nullptr);
}

size_t cf_stitch_batchnorm_workspace_size(int64_t rows, int64_t cols) {
    (void)rows;
    (void)cols;
    // under either mapping (the Global one may be forced for any shape): error
    // word, arrive/depart counters, one float2 partial per CTA and strip column
    return cf::kErrBytes + 256 + size_t(cf::kBnMaxGlobalCtas) * 128 * sizeof(float2);
}

// BatchNorm mapping ([AStitch] "Four stitching schemes", "Adaptive thread
// mapping"): Regional when one CTA can hold every row of its columns,
// otherwise Global -- one resident wave of CTAs (vertical packing) meeting at
// an in-kernel barrier, as many row chunks per column strip as fit.
static cf_status plan_batchnorm(int64_t rows, int64_t cols, const cf_tuning &t, const cf::DeviceInfo &dev,
                                cf::BnPlan *pp) {
    cf::BnPlan &p = *pp;
    p.pdl = t.disable_pdl == 0;
    p.timeout_ns = 1000ull * (t.timeout_us ? t.timeout_us : kDefaultTimeoutUs);
    p.extra_arrivals = t.extra_arrivals;
    const int ng = int((cols + 3) / 4);
    int mapping = t.stitch_mapping;
    if (mapping == 0) mapping = rows <= cf::kBnRegionalMaxRows ? 3 : 4;
    if (mapping == 5 || mapping == 6) mapping = 4;  // Global without TMA streaming (5) or with tiled copies (6)
    if (mapping == 3) {
        if (rows > cf::kBnRegionalMaxRows) return CF_ERR_UNSUPPORTED;
        p.mapping = 3;
        p.rpt = next_pow2(int((rows + 7) / 8));
        p.grid = (ng + 31) / 32;
        return CF_OK;
    }
    if (mapping != 4) return CF_ERR_INVALID_ARG;
    p.mapping = 4;
    p.lpr = std::min(32, next_pow2(ng));
    p.strips = (ng + p.lpr - 1) / p.lpr;
    // 128-bit rows stream through shared memory by TMA (rows addressable as int32)
    p.tma = p.vec && t.stitch_mapping != 5 && rows < (int64_t(1) << 31);
    int bps = p.tma ? cf::bn_tma_blocks_per_sm(p.lpr) : cf::bn_global_blocks_per_sm(p.lpr, p.vec);
    if (bps <= 0) return CF_ERR_NOT_RESIDENT;
    int cap = std::min(dev.sm_count * bps, cf::kBnMaxGlobalCtas);
    if (t.max_clusters > 0) cap = std::min(cap, int(t.max_clusters));
    if (p.strips > cap) return CF_ERR_UNSUPPORTED;
    int chunks = cap / p.strips;
    // a chunk of at least 32 rows per CTA (fewer chunks for short columns)
    chunks = int(std::max<int64_t>(1, std::min<int64_t>(chunks, rows / 32)));
    p.grid = chunks * p.strips;
    if (p.tma) {  // chunk boundaries on stage boundaries: no two CTAs store the same rows
        const int br = cf::bn_tma_box_rows(p.lpr);
        const int64_t per = (rows + chunks - 1) / chunks;
        p.rows_per_chunk = ((per + br - 1) / br) * br;
    }
    return CF_OK;
}

cf_status cf_stitch_batchnorm_ex(const float *A, const float *gamma, const float *beta, float *out,
                                 float *mean_out, float *var_out, int64_t rows, int64_t cols, float eps, void *ws,
                                 size_t ws_bytes, cf_stream_t stream, const cf_tuning *tuning) {
    if (rows < 0 || cols < 0) return CF_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CF_OK;
    if (!A || !gamma || !beta || !out || !ws) return CF_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(gamma) |
         reinterpret_cast<uintptr_t>(beta) | reinterpret_cast<uintptr_t>(mean_out) |
         reinterpret_cast<uintptr_t>(var_out)) & 3u)
        return CF_ERR_MISALIGNED;
    if (!aligned16(ws)) return CF_ERR_MISALIGNED;
    if (cols > (int64_t(1) << 30) || rows > (int64_t(1) << 40)) return CF_ERR_UNSUPPORTED;
    if (ws_bytes < cf_stitch_batchnorm_workspace_size(rows, cols)) return CF_ERR_WORKSPACE_TOO_SMALL;
    cf_tuning tz;
    cf_tuning_default(&tz);
    const cf_tuning &t = tuning ? *tuning : tz;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;
    cf::BnPlan p;
    p.vec = (cols % 4 == 0) && aligned16(A) && aligned16(out);
    cf_status st = plan_batchnorm(rows, cols, t, dev, &p);
    if (st != CF_OK) return st;
    if (p.mapping == 4 && ws_bytes < cf::kErrBytes + 256 + size_t(p.grid) * 4 * p.lpr * sizeof(float2))
        return CF_ERR_WORKSPACE_TOO_SMALL;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    if (p.mapping == 4 && p.tma) {
        cf::BnTmaArgs a;
        std::memset(&a, 0, sizeof(a));
        const uint32_t W = uint32_t(4 * p.lpr), br = uint32_t(cf::bn_tma_box_rows(p.lpr));
        if (!make_tmap_f32(&a.tmap_a, A, uint64_t(rows), uint64_t(cols), W, br)) return CF_ERR_CUDA;
        a.gamma = gamma;
        a.beta = beta;
        a.mean_out = mean_out;
        a.var_out = var_out;
        a.err = reinterpret_cast<uint32_t *>(wsb);
        a.counters = reinterpret_cast<uint32_t *>(wsb + cf::kErrBytes);
        a.partials = reinterpret_cast<float2 *>(wsb + cf::kErrBytes + 256);
        a.rows = rows;
        a.cols = int(cols);
        a.strips = p.strips;
        a.rows_per_chunk = int(p.rows_per_chunk);
        a.extra_arrivals = p.extra_arrivals;
        a.eps = eps;
        a.timeout_ns = p.timeout_ns;
        a.trace = reinterpret_cast<unsigned long long *>(t.trace);
        a.A = A;
        a.out = out;
        a.flat = (cols == int64_t(W) && t.stitch_mapping != 6) ? 1 : 0;  // 6: tiled copies forced (comparison)
        cf::bn_tma_buffers(p.lpr, t.stages, &a.ring, &a.res);
        cudaError_t e = cf::launch_batchnorm_tma(p.lpr, a, p.grid, p.pdl, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e);
        return CF_OK;
    }
    cudaError_t e = cf::launch_batchnorm(p, A, gamma, beta, out, mean_out, var_out, rows, cols, eps,
                                         reinterpret_cast<uint32_t *>(wsb),
                                         reinterpret_cast<uint32_t *>(wsb + cf::kErrBytes),
                                         reinterpret_cast<float2 *>(wsb + cf::kErrBytes + 256),
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return CF_OK;
}

cf_status cf_stitch_batchnorm(const float *A, const float *gamma, const float *beta, float *out, float *mean_out,
                              float *var_out, int64_t rows, int64_t cols, float eps, void *ws, size_t ws_bytes,
                              cf_stream_t stream) {
    return cf_stitch_batchnorm_ex(A, gamma, beta, out, mean_out, var_out, rows, cols, eps, ws, ws_bytes, stream,
                                  nullptr);
}

cf_status cf_query_stitch_batchnorm_plan(int64_t rows, int64_t cols, const cf_tuning *tuning, int32_t *mapping,
                                         int32_t *grid) {
    if (rows <= 0 || cols <= 0 || !mapping || !grid) return CF_ERR_INVALID_ARG;
    cf_tuning tz;
    cf_tuning_default(&tz);
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;
    cf::BnPlan p;
    p.vec = cols % 4 == 0;
    cf_status st = plan_batchnorm(rows, cols, tuning ? *tuning : tz, dev, &p);
    *mapping = p.mapping;
    *grid = p.grid;
    return st;
}

// -------------------------------------------------------------------------
// fused GEMM
// -------------------------------------------------------------------------
// residency of every candidate cluster size at the shared memory it would use
static cf_status device_plan(int kind, int64_t M, int64_t N, int64_t K, const cf_tuning *tuning,
                             const cf::DeviceInfo &dev, cf_plan *plan, int32_t active[17]) {
    cf_tuning tz;
    cf_tuning_default(&tz);
    const cf_tuning &t = tuning ? *tuning : tz;
    if (N <= 0 || K <= 0 || N % 64 != 0 || K % 64 != 0) return CF_ERR_UNSUPPORTED;
    // residency is queried at the narrow tile's shared memory; a wide tile's is
    // also above half of the SM's, so it is one CTA per SM all the same
    int ns = t.n_slice ? t.n_slice : ((N % 256 == 0) ? 256 : (N % 128 == 0) ? 128 : 64);
    if ((ns != 64 && ns != 128 && ns != 256 && ns != 512) || N % ns != 0) return CF_ERR_UNSUPPORTED;
    if (ns == 512) ns = 256;
    // too few tiles to give every SM one: the planner also weighs narrower
    // tiles, whose cluster sizes divide N / 64
    if (t.n_slice == 0 && ((M + cf::kBlockM - 1) / cf::kBlockM) * (N / ns) < dev.sm_count) ns = 64;
    const int64_t cpr = N / ns;
    for (int c = 0; c <= 16; ++c) active[c] = 0;
    // residency is per SM (one CTA per SM at any of these shared-memory
    // sizes), so one query per total cluster size serves every (C_N, C_M)
    for (int c = 1; c <= 16; ++c) {
        const bool as_cn = (cpr % c == 0);
        const bool as_pair = (c % 2 == 0) && (cpr % (c / 2) == 0) && ns >= 128;
        if (!as_cn && !as_pair) continue;
        const int cn = as_cn ? c : c / 2;
        const int st = gemm_stages_for(ns, cn, t.stages, !as_cn, true);
        const int smem = cf::gemm_fused_smem_bytes(st, cn, ns, !as_cn, true, 1);
        if (smem > std::min(kMaxSmem, dev.max_smem_optin)) continue;
        active[c] = max_active_cached(dev.device, kind, !as_cn, c, smem);
    }
    return cf_plan_gemm_fused(M, N, K, dev.sm_count, active, tuning, plan);
}

cf_status cf_query_gemm_fused_plan(int64_t M, int64_t N, int64_t K, int32_t kind, const cf_tuning *tuning,
                                   cf_plan *plan, int32_t max_active_clusters[17]) {
    if (!plan || kind < 0 || kind > 2 || M < 0) return CF_ERR_INVALID_ARG;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;
    int32_t active[17];
    cf_status st = device_plan(kind, M, N, K, tuning, dev, plan, active);
    if (max_active_clusters)
        for (int c = 0; c <= 16; ++c) max_active_clusters[c] = active[c];
    return st;
}

static cf_status gemm_fused_common(int kind, const void *X, const void *W, const float *bias, const float *gamma,
                                   const float *beta, void *Y, int64_t M, int64_t N, int64_t K, float alpha,
                                   float eps, void *ws, size_t ws_bytes, cf_stream_t stream,
                                   const cf_tuning *tuning, int rms = 0, const void *R = nullptr,
                                   long long mask_offset = 0) {
    if (M < 0 || N <= 0 || K <= 0) return CF_ERR_INVALID_ARG;
    if (!X || !W || !Y || !ws) return CF_ERR_INVALID_ARG;
    const bool sm = kind == cf::EPI_SOFTMAX || kind == cf::EPI_SOFTMAX_MASK;
    if (!sm && (!gamma || (!beta && !rms))) return CF_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || (bias && !aligned16(bias)) ||
        (gamma && !aligned16(gamma)) || (beta && !aligned16(beta)) || (R && !aligned16(R)))
        return CF_ERR_MISALIGNED;
    if (R && (R == X || R == W)) return CF_ERR_INVALID_ARG;
    if (K % 64 != 0 || N % 64 != 0) return CF_ERR_UNSUPPORTED;
    if (ws_bytes < cf_gemm_fused_workspace_size(M, N, K)) return CF_ERR_WORKSPACE_TOO_SMALL;
    if (M == 0) return CF_OK;
    cf_tuning tz;
    cf_tuning_default(&tz);
    const cf_tuning &t = tuning ? *tuning : tz;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;

    cf_plan plan;
    int32_t active[17];
    cf_status st = device_plan(kind, M, N, K, tuning, dev, &plan, active);
    if (st != CF_OK) return st;

    cf::GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!make_tmap_bf16(&a.tmap_x, X, uint64_t(M), uint64_t(K), 64, 128)) return CF_ERR_CUDA;
    if (!make_tmap_w(&a.tmap_w, W, uint64_t(K), uint64_t(N), w_blocks(plan.n_slice, plan.cluster_m)))
        return CF_ERR_CUDA;
    if (!make_tmap_bf16(&a.tmap_y, Y, uint64_t(M), uint64_t(N), 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) return CF_ERR_CUDA;
    a.bias = bias;
    a.gamma = gamma;
    a.beta = beta;
    a.y = static_cast<uint16_t *>(Y);
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    a.err = reinterpret_cast<uint32_t *>(wsb);
    a.counters = reinterpret_cast<uint32_t *>(wsb + cf::kErrBytes);
    {
        const size_t rba = size_t((plan.row_blocks + plan.cluster_m - 1) / plan.cluster_m) * plan.cluster_m;
        a.partials = reinterpret_cast<float2 *>(wsb + cf::kErrBytes + cf::align_up(8 * rba, 256));
    }
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.alpha = alpha;
    a.eps = eps;
    a.n_slice = plan.n_slice;
    a.cluster = plan.cluster_size;
    a.cluster_m = plan.cluster_m;
    a.groups = plan.groups;
    a.leader = plan.leader_mode;
    a.row_blocks = plan.row_blocks;
    a.super_blocks = (plan.row_blocks + plan.cluster_m - 1) / plan.cluster_m;
    a.row_blocks_alloc = a.super_blocks * plan.cluster_m;
    a.extra_arrivals = t.extra_arrivals;
    a.rms = rms;
    a.resid = static_cast<const uint16_t *>(R);
    a.mask_offset = mask_offset;
    a.timeout_ns = 1000ull * (t.timeout_us ? t.timeout_us : kDefaultTimeoutUs);
    a.trace = reinterpret_cast<unsigned long long *>(t.trace);
    a.stg_bufs = plan.staging_buffers;
    cudaError_t e = cf::launch_gemm_fused(kind, a, plan.clusters, plan.stages, plan.smem_bytes, t.disable_pdl == 0,
                                          reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return CF_OK;
}

cf_status cf_gemm_fused_rownorm_ex(const void *X, const void *W, const float *bias, const float *gamma,
                                   const float *beta, void *Y, int64_t M, int64_t N, int64_t K, float alpha,
                                   float eps, cf_activation act, void *ws, size_t ws_bytes, cf_stream_t stream,
                                   const cf_tuning *tuning) {
    int kind;
    if (act == CF_ACT_NONE) kind = cf::EPI_LN;
    else if (act == CF_ACT_GELU_TANH) kind = cf::EPI_GELU_LN;
    else return CF_ERR_INVALID_ARG;
    return gemm_fused_common(kind, X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, ws, ws_bytes, stream, tuning);
}

cf_status cf_gemm_fused_rownorm(const void *X, const void *W, const float *bias, const float *gamma,
                                const float *beta, void *Y, int64_t M, int64_t N, int64_t K, float alpha,
                                float eps, cf_activation act, void *ws, size_t ws_bytes, cf_stream_t stream) {
    return cf_gemm_fused_rownorm_ex(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, act, ws, ws_bytes, stream,
                                    nullptr);
}

cf_status cf_gemm_fused_rmsnorm_ex(const void *X, const void *W, const float *bias, const float *gamma,
                                   const float *beta, void *Y, int64_t M, int64_t N, int64_t K, float alpha,
                                   float eps, cf_activation act, void *ws, size_t ws_bytes, cf_stream_t stream,
                                   const cf_tuning *tuning) {
    int kind;
    if (act == CF_ACT_NONE) kind = cf::EPI_LN;
    else if (act == CF_ACT_GELU_TANH) kind = cf::EPI_GELU_LN;
    else return CF_ERR_INVALID_ARG;
    return gemm_fused_common(kind, X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, ws, ws_bytes, stream, tuning,
                             1);
}

cf_status cf_gemm_fused_rmsnorm(const void *X, const void *W, const float *bias, const float *gamma,
                                const float *beta, void *Y, int64_t M, int64_t N, int64_t K, float alpha,
                                float eps, cf_activation act, void *ws, size_t ws_bytes, cf_stream_t stream) {
    return cf_gemm_fused_rmsnorm_ex(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, act, ws, ws_bytes, stream,
                                    nullptr);
}

cf_status cf_gemm_fused_residual_norm_ex(const void *X, const void *W, const float *bias, const void *R,
                                         const float *gamma, const float *beta, void *Y, int64_t M, int64_t N,
                                         int64_t K, float alpha, float eps, cf_activation act, cf_norm norm,
                                         void *ws, size_t ws_bytes, cf_stream_t stream, const cf_tuning *tuning) {
    int kind;
    if (act == CF_ACT_NONE) kind = cf::EPI_LN;
    else if (act == CF_ACT_GELU_TANH) kind = cf::EPI_GELU_LN;
    else return CF_ERR_INVALID_ARG;
    if (norm != CF_NORM_LAYER && norm != CF_NORM_RMS) return CF_ERR_INVALID_ARG;
    if (!R) return CF_ERR_INVALID_ARG;
    return gemm_fused_common(kind, X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, ws, ws_bytes, stream, tuning,
                             norm == CF_NORM_RMS ? 1 : 0, R);
}

cf_status cf_gemm_fused_residual_norm(const void *X, const void *W, const float *bias, const void *R,
                                      const float *gamma, const float *beta, void *Y, int64_t M, int64_t N,
                                      int64_t K, float alpha, float eps, cf_activation act, cf_norm norm, void *ws,
                                      size_t ws_bytes, cf_stream_t stream) {
    return cf_gemm_fused_residual_norm_ex(X, W, bias, R, gamma, beta, Y, M, N, K, alpha, eps, act, norm, ws,
                                          ws_bytes, stream, nullptr);
}

cf_status cf_gemm_fused_rowsoftmax_ex(const void *X, const void *W, const float *bias, void *Y, int64_t M,
                                      int64_t N, int64_t K, float scale, void *ws, size_t ws_bytes,
                                      cf_stream_t stream, const cf_tuning *tuning) {
    return gemm_fused_common(cf::EPI_SOFTMAX, X, W, bias, nullptr, nullptr, Y, M, N, K, scale, 0.f, ws, ws_bytes,
                             stream, tuning);
}

cf_status cf_gemm_fused_rowsoftmax_causal_ex(const void *X, const void *W, const float *bias, void *Y, int64_t M,
                                             int64_t N, int64_t K, float scale, int64_t offset, void *ws,
                                             size_t ws_bytes, cf_stream_t stream, const cf_tuning *tuning) {
    return gemm_fused_common(cf::EPI_SOFTMAX_MASK, X, W, bias, nullptr, nullptr, Y, M, N, K, scale, 0.f, ws,
                             ws_bytes, stream, tuning, 0, nullptr, (long long)offset);
}

cf_status cf_gemm_fused_rowsoftmax_causal(const void *X, const void *W, const float *bias, void *Y, int64_t M,
                                          int64_t N, int64_t K, float scale, int64_t offset, void *ws,
                                          size_t ws_bytes, cf_stream_t stream) {
    return cf_gemm_fused_rowsoftmax_causal_ex(X, W, bias, Y, M, N, K, scale, offset, ws, ws_bytes, stream,
                                              nullptr);
}

cf_status cf_gemm_fused_rowsoftmax(const void *X, const void *W, const float *bias, void *Y, int64_t M, int64_t N,
                                   int64_t K, float scale, void *ws, size_t ws_bytes, cf_stream_t stream) {
    return cf_gemm_fused_rowsoftmax_ex(X, W, bias, Y, M, N, K, scale, ws, ws_bytes, stream, nullptr);
}

// -------------------------------------------------------------------------
// back-to-back GEMM
// -------------------------------------------------------------------------
size_t cf_b2b_workspace_size(void) { return cf::kB2bWorkspaceBytes; }

static int b2b_active_cached(int device, int op, int cluster, int n2, int smem) {
    static std::map<std::tuple<int, int, int, int, int>, int> cache;
    auto key = std::make_tuple(device, op, cluster, n2, smem);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = cf::b2b_max_active_clusters(op, cluster, n2, smem);
    std::lock_guard<std::mutex> lk(g_mu);
    cache[key] = n;
    return n;
}

// B2B kernel choice: the cluster kernel (C = N1/256 CTAs per row block, the
// intermediate's columns partitioned over the cluster, partial outputs
// reduce-scattered) or the stream kernel (one CTA per row block, N1 streamed
// in 256-column chunks; LayerNorm in one pass).  tuning->n_slice selects:
// 0 auto, 128 stream, 256 cluster (the plan reports the same values).
static cf_status b2b_plan(int64_t M, int64_t K, int64_t N1, int64_t N2, int op, const cf_tuning *tuning,
                          const cf::DeviceInfo &dev, cf_plan *plan) {
    if (M < 0 || K <= 0 || N1 <= 0 || N2 <= 0) return CF_ERR_INVALID_ARG;
    if (op != CF_B2B_SOFTMAX && op != CF_B2B_GELU_TANH && op != CF_B2B_LAYERNORM) return CF_ERR_INVALID_ARG;
    if (K % 8 != 0 || N1 % 256 != 0 || (N2 != 64 && N2 != 128)) return CF_ERR_UNSUPPORTED;
    if (M > (int64_t(1) << 31) - 128 || K > (int64_t(1) << 30) || N1 > (int64_t(1) << 30)) return CF_ERR_UNSUPPORTED;
    const int64_t C = N1 / 256;
    const bool cluster_ok = C == 1 || C == 2 || C == 4 || C == 8;
    const int reqn = tuning ? tuning->n_slice : 0;
    bool stream;
    // one CTA per row block: no cluster exchange at all
    if (reqn == 0) stream = true;
    else if (reqn == 128) stream = true;
    else if (reqn == 256) stream = false;
    else return CF_ERR_UNSUPPORTED;
    if (!stream && !cluster_ok) return CF_ERR_UNSUPPORTED;
    const int req = tuning ? tuning->stages : 0;
    if (req < 0 || req > 6) return CF_ERR_UNSUPPORTED;
    std::memset(plan, 0, sizeof(*plan));
    plan->groups = 1;
    plan->cluster_m = 1;
    plan->row_blocks = int32_t((M + 127) / 128);
    if (stream) {
        // the ring depth is fixed per mode (tuning->stages does not apply); at
        // least half the SM's shared memory, so that one CTA (with all 512
        // tensor-memory columns) runs per SM
        const int stages = cf::b2b_stream_stages(op, int(K));
        const int smem = std::max(cf::b2b_stream_smem_bytes(op, int(K)), kMaxSmem / 2 + 1024);
        if (smem > kMaxSmem || smem > dev.max_smem_optin) return CF_ERR_UNSUPPORTED;
        plan->n_slice = 128;  // the stream kernel's selector value (its chunks are 256 columns)
        plan->ctas_per_row = 1;
        plan->cluster_size = 1;
        plan->stages = stages;
        plan->smem_bytes = smem;
        int ctas = int(std::min<int64_t>(plan->row_blocks, dev.sm_count));
        if (tuning && tuning->max_clusters > 0) ctas = std::min(ctas, int(tuning->max_clusters));
        plan->clusters = ctas;
        return CF_OK;
    }
    int stages = req > 0 ? req : 4;
    while (stages > 2 && cf::b2b_smem_bytes(stages, int(C), int(N2), op) > kMaxSmem) --stages;
    const int smem = cf::b2b_smem_bytes(stages, int(C), int(N2), op);
    if (smem > kMaxSmem || smem > dev.max_smem_optin) return CF_ERR_UNSUPPORTED;
    plan->n_slice = 256;
    plan->ctas_per_row = int32_t(C);
    plan->cluster_size = int32_t(C);
    plan->stages = stages;
    plan->smem_bytes = smem;
    const int active = b2b_active_cached(dev.device, op, int(C), int(N2), smem);
    if (active <= 0) return CF_ERR_NOT_RESIDENT;
    int clusters = std::min<int64_t>(plan->row_blocks, active);
    if (tuning && tuning->max_clusters > 0) clusters = std::min(clusters, int(tuning->max_clusters));
    plan->clusters = clusters;
    return CF_OK;
}

cf_status cf_query_b2b_plan(int64_t M, int64_t K, int64_t N1, int64_t N2, cf_b2b_op op, const cf_tuning *tuning,
                            cf_plan *plan) {
    if (!plan) return CF_ERR_INVALID_ARG;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;
    return b2b_plan(M, K, N1, N2, int(op), tuning, dev, plan);
}

static cf_status b2b_common(const void *X, const void *W1, const float *b1, const float *gamma1,
                            const float *beta1, const void *W2, void *O, int64_t M, int64_t K, int64_t N1,
                            int64_t N2, float alpha, float eps, int op, void *ws, size_t ws_bytes,
                            cf_stream_t stream, const cf_tuning *tuning) {
    if (M < 0 || K <= 0 || N1 <= 0 || N2 <= 0) return CF_ERR_INVALID_ARG;
    if (op != CF_B2B_SOFTMAX && op != CF_B2B_GELU_TANH && op != CF_B2B_LAYERNORM) return CF_ERR_INVALID_ARG;
    if (!X || !W1 || !W2 || !O || !ws) return CF_ERR_INVALID_ARG;
    if (op == CF_B2B_LAYERNORM && (!gamma1 || !beta1)) return CF_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W2) || !aligned16(O) || (b1 && !aligned16(b1)) ||
        (gamma1 && !aligned16(gamma1)) || (beta1 && !aligned16(beta1)))
        return CF_ERR_MISALIGNED;
    if (O == X || O == W1 || O == W2) return CF_ERR_INVALID_ARG;
    if (K % 8 != 0 || N1 % 256 != 0 || (N2 != 64 && N2 != 128)) return CF_ERR_UNSUPPORTED;
    if (ws_bytes < cf_b2b_workspace_size()) return CF_ERR_WORKSPACE_TOO_SMALL;
    if (M == 0) return CF_OK;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;
    cf_plan plan;
    cf_status st = b2b_plan(M, K, N1, N2, op, tuning, dev, &plan);
    if (st != CF_OK) return st;

    cf::B2bArgs a;
    std::memset(&a, 0, sizeof(a));
    const bool stream_kernel = plan.cluster_size == 1 && plan.n_slice == 128;
    if (!make_tmap_bf16(&a.tmap_x, X, uint64_t(M), uint64_t(K), 64, 128)) return CF_ERR_CUDA;
    if (!make_tmap_w(&a.tmap_w1, W1, uint64_t(K), uint64_t(N1), 4)) return CF_ERR_CUDA;  // 256 columns
    if (!make_tmap_w(&a.tmap_w2, W2, uint64_t(N1), uint64_t(N2), uint32_t(N2 / 64), stream_kernel ? 128 : 64))
        return CF_ERR_CUDA;
    if (stream_kernel &&
        !make_tmap_bf16(&a.tmap_o, O, uint64_t(M), uint64_t(N2), 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return CF_ERR_CUDA;
    a.b1 = b1;
    a.gamma1 = gamma1;
    a.beta1 = beta1;
    a.eps = eps;
    a.out = static_cast<uint16_t *>(O);
    a.err = static_cast<uint32_t *>(ws);
    a.M = int(M);
    a.K = int(K);
    a.N1 = int(N1);
    a.N2 = int(N2);
    a.cluster = plan.cluster_size;
    a.alpha = alpha;
    const uint32_t tus = tuning && tuning->timeout_us ? tuning->timeout_us : kDefaultTimeoutUs;
    a.timeout_ns = 1000ull * tus;
    a.trace = tuning ? reinterpret_cast<unsigned long long *>(tuning->trace) : nullptr;
    a.extra_arrivals = tuning && tuning->extra_arrivals > 0 ? tuning->extra_arrivals : 0;
    const bool pdl = !(tuning && tuning->disable_pdl);
    if (stream_kernel && op == CF_B2B_LAYERNORM) {
        // the LayerNorm output terms gamma1^T W2 and beta1^T W2, read by the
        // stream kernel once its row statistics are known
        a.fold = reinterpret_cast<const float *>(static_cast<unsigned char *>(ws) + cf::kB2bFoldOff);
        cudaError_t ef = cf::launch_b2b_ln_fold(W2, gamma1, beta1, int(N1), int(N2), static_cast<unsigned char *>(ws),
                                                pdl, reinterpret_cast<cudaStream_t>(stream));
        if (ef != cudaSuccess) return cuda_fail(ef);
    }
    cudaError_t e = stream_kernel ? cf::launch_b2b_stream(op, a, plan.clusters, plan.smem_bytes, pdl,
                                                          reinterpret_cast<cudaStream_t>(stream))
                                  : cf::launch_b2b(op, a, plan.clusters, plan.stages, plan.smem_bytes, pdl,
                                                   reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return CF_OK;
}

cf_status cf_b2b_gemm_ex(const void *X, const void *W1, const float *b1, const void *W2, void *O, int64_t M,
                         int64_t K, int64_t N1, int64_t N2, float alpha, cf_b2b_op op, void *ws, size_t ws_bytes,
                         cf_stream_t stream, const cf_tuning *tuning) {
    if (op == CF_B2B_LAYERNORM) return CF_ERR_INVALID_ARG;  // needs gamma1, beta1: cf_b2b_gemm_layernorm
    return b2b_common(X, W1, b1, nullptr, nullptr, W2, O, M, K, N1, N2, alpha, 0.f, int(op), ws, ws_bytes, stream,
                      tuning);
}

cf_status cf_b2b_gemm(const void *X, const void *W1, const float *b1, const void *W2, void *O, int64_t M, int64_t K,
                      int64_t N1, int64_t N2, float alpha, cf_b2b_op op, void *ws, size_t ws_bytes,
                      cf_stream_t stream) {
    return cf_b2b_gemm_ex(X, W1, b1, W2, O, M, K, N1, N2, alpha, op, ws, ws_bytes, stream, nullptr);
}

cf_status cf_b2b_gemm_layernorm_ex(const void *X, const void *W1, const float *b1, const float *gamma1,
                                   const float *beta1, const void *W2, void *O, int64_t M, int64_t K, int64_t N1,
                                   int64_t N2, float alpha, float eps, void *ws, size_t ws_bytes, cf_stream_t stream,
                                   const cf_tuning *tuning) {
    return b2b_common(X, W1, b1, gamma1, beta1, W2, O, M, K, N1, N2, alpha, eps, CF_B2B_LAYERNORM, ws, ws_bytes,
                      stream, tuning);
}

cf_status cf_b2b_gemm_layernorm(const void *X, const void *W1, const float *b1, const float *gamma1,
                                const float *beta1, const void *W2, void *O, int64_t M, int64_t K, int64_t N1,
                                int64_t N2, float alpha, float eps, void *ws, size_t ws_bytes, cf_stream_t stream) {
    return cf_b2b_gemm_layernorm_ex(X, W1, b1, gamma1, beta1, W2, O, M, K, N1, N2, alpha, eps, ws, ws_bytes, stream,
                                    nullptr);
}

}  // extern "C"

// =========================================================================
// Variant of the fused GEMM + LayerNorm call that allocates nothing and takes
// no workspace argument.  Its scratch (error word, barrier counters, global
// partials) is one file-scope device array of fixed size that every device
// loading this library holds until the process exits.  Host code may not use
// the array's name as a device address: the address is looked up once per
// device with cudaGetSymbolAddress (that device current) and passed to the
// kernel like any workspace pointer.
// =========================================================================
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on `device` (the current device),
// looked up on the first call for that device and cached.
static cf_status noalloc_scratch(int device, void **out) {
    static void *addr[64] = {};
    if (device < 0 || device >= 64) return CF_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (addr[device] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            g_last_cuda_error = int(e);
            return CF_ERR_CUDA;
        }
        addr[device] = p;
    }
    *out = addr[device];
    return CF_OK;
}

extern "C" cf_status cf_gemm_fused_rownorm_noalloc(const void *X, const void *W, const float *bias,
                                                   const float *gamma, const float *beta, void *Y, int64_t M,
                                                   int64_t N, int64_t K, float alpha, float eps,
                                                   cf_activation act, cf_stream_t stream) {
    int kind;
    if (act == CF_ACT_NONE) kind = cf::EPI_LN;
    else if (act == CF_ACT_GELU_TANH) kind = cf::EPI_GELU_LN;
    else return CF_ERR_INVALID_ARG;
    if (M < 0 || N <= 0 || K <= 0) return CF_ERR_INVALID_ARG;
    if (!X || !W || !Y || !gamma || !beta) return CF_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || (bias && !aligned16(bias)) || !aligned16(gamma) ||
        !aligned16(beta))
        return CF_ERR_MISALIGNED;
    if (K % 64 != 0 || N % 64 != 0) return CF_ERR_UNSUPPORTED;
    if (M == 0) return CF_OK;
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;

    cf_plan plan;
    int32_t active[17];
    cf_status st = device_plan(kind, M, N, K, nullptr, dev, &plan, active);
    if (st != CF_OK) return st;
    // scratch this launch uses: error word + counters (must start at zero) and
    // one float2 per row and cluster group of the global partial buffer
    const size_t rba = size_t((plan.row_blocks + plan.cluster_m - 1) / plan.cluster_m) * plan.cluster_m;
    const size_t head = cf::kErrBytes + cf::align_up(8 * rba, 256);
    const size_t gp = size_t(plan.groups) + size_t(plan.groups & 1);
    const size_t need = head + rba * gp * 128 * sizeof(float2);
    if (need > kNoAllocScratchBytes) return CF_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    st = noalloc_scratch(dev.device, &scratch);
    if (st != CF_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(scratch, 0, head, s);
    if (e != cudaSuccess) return cuda_fail(e);

    cf::GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!make_tmap_bf16(&a.tmap_x, X, uint64_t(M), uint64_t(K), 64, 128)) return CF_ERR_CUDA;
    if (!make_tmap_w(&a.tmap_w, W, uint64_t(K), uint64_t(N), w_blocks(plan.n_slice, plan.cluster_m)))
        return CF_ERR_CUDA;
    if (!make_tmap_bf16(&a.tmap_y, Y, uint64_t(M), uint64_t(N), 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) return CF_ERR_CUDA;
    uint8_t *sb = static_cast<uint8_t *>(scratch);
    a.bias = bias;
    a.gamma = gamma;
    a.beta = beta;
    a.y = static_cast<uint16_t *>(Y);
    a.err = reinterpret_cast<uint32_t *>(sb);
    a.counters = reinterpret_cast<uint32_t *>(sb + cf::kErrBytes);
    a.partials = reinterpret_cast<float2 *>(sb + head);
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.alpha = alpha;
    a.eps = eps;
    a.n_slice = plan.n_slice;
    a.cluster = plan.cluster_size;
    a.cluster_m = plan.cluster_m;
    a.groups = plan.groups;
    a.leader = plan.leader_mode;
    a.row_blocks = plan.row_blocks;
    a.super_blocks = (plan.row_blocks + plan.cluster_m - 1) / plan.cluster_m;
    a.row_blocks_alloc = a.super_blocks * plan.cluster_m;
    a.extra_arrivals = 0;
    a.timeout_ns = 1000ull * kDefaultTimeoutUs;
    a.stg_bufs = plan.staging_buffers;
    e = cf::launch_gemm_fused(kind, a, plan.clusters, plan.stages, plan.smem_bytes, true, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return CF_OK;
}

extern "C" cf_status cf_gemm_fused_rownorm_noalloc_status(cf_stream_t stream, int32_t *info) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e);
    void *scratch = nullptr;
    cf_status st = noalloc_scratch(device, &scratch);
    if (st != CF_OK) return st;
    return cf_get_device_status(scratch, stream, info);
}

// =========================================================================
// The unfused two-kernel composition (a measured baseline, not a fallback):
// GEMM -> fp32 P in global memory -> row kernel.  Same results within the
// fused calls' tolerances; it pays the intermediate's write and read.
// =========================================================================
namespace {

size_t unfused_p_bytes(int64_t M, int64_t N) { return cf::align_up(size_t(M) * size_t(N) * 4, 256); }

// P = X . W (fp32), with the fused kernel's store-only epilogue: every tile
// is independent (no row reduction), so any resident cluster count works.
cf_status gemm_store_f32(const void *X, const void *W, float *P, uint32_t *err, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream) {
    cf::DeviceInfo dev;
    if (!cf::current_device_info(&dev)) return CF_ERR_NO_DEVICE;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return CF_ERR_NO_DEVICE;
    const int ns = (N % 256 == 0) ? 256 : (N % 128 == 0) ? 128 : 64;
    const int cpr = int(N / ns);
    const int rb = int((M + cf::kBlockM - 1) / cf::kBlockM);
    const int nk = int(K / 64);
    const int cm = (nk >= 8 && rb >= 2 && ns >= 128) ? 2 : 1;
    const bool pair = cm == 2;
    const int stages = gemm_stages_for(ns, 1, 0, pair, false, 1);
    int sb = 1;
    if (cf::gemm_fused_smem_bytes(stages, 1, ns, pair, false, 2) <= kMaxSmem) sb = 2;
    const int smem = cf::gemm_fused_smem_bytes(stages, 1, ns, pair, false, sb);
    const int active = max_active_cached(dev.device, cf::EPI_STORE_F32, pair, cm, smem);
    if (active <= 0) return CF_ERR_NOT_RESIDENT;
    const int sblocks = (rb + cm - 1) / cm;
    const int64_t tickets = int64_t(sblocks) * cpr;
    const int clusters = int(std::min<int64_t>(active, tickets));

    cf::GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!make_tmap_bf16(&a.tmap_x, X, uint64_t(M), uint64_t(K), 64, 128)) return CF_ERR_CUDA;
    if (!make_tmap_w(&a.tmap_w, W, uint64_t(K), uint64_t(N), w_blocks(ns, cm))) return CF_ERR_CUDA;
    if (!make_tmap_f32_store(&a.tmap_y, P, uint64_t(M), uint64_t(N))) return CF_ERR_CUDA;
    a.err = err;
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.alpha = 1.f;
    a.n_slice = ns;
    a.cluster = 1;
    a.cluster_m = cm;
    a.groups = cpr;  // tickets enumerate every tile of a row block
    a.row_blocks = rb;
    a.super_blocks = sblocks;
    a.row_blocks_alloc = sblocks * cm;
    a.timeout_ns = 1000ull * kDefaultTimeoutUs;
    a.stg_bufs = sb;
    cudaError_t e = cf::launch_gemm_fused(cf::EPI_STORE_F32, a, clusters, stages, smem, true, stream);
    return e == cudaSuccess ? CF_OK : cuda_fail(e);
}

cf_status unfused_common(int op, const void *X, const void *W, const float *bias, const float *gamma,
                         const float *beta, void *Y, int64_t M, int64_t N, int64_t K, float alpha, float eps,
                         void *ws, size_t ws_bytes, cf_stream_t stream, int rms = 0, const void *R = nullptr) {
    if (M < 0 || N <= 0 || K <= 0) return CF_ERR_INVALID_ARG;
    if (!X || !W || !Y || !ws) return CF_ERR_INVALID_ARG;
    if (op != 2 && (!gamma || (!beta && !rms))) return CF_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || !aligned16(ws) || (bias && !aligned16(bias)) ||
        (gamma && !aligned16(gamma)) || (beta && !aligned16(beta)) || (R && !aligned16(R)))
        return CF_ERR_MISALIGNED;
    if (K % 64 != 0 || N % 64 != 0 || N > 256 * 64) return CF_ERR_UNSUPPORTED;
    if (ws_bytes < cf_unfused_workspace_size(M, N, K)) return CF_ERR_WORKSPACE_TOO_SMALL;
    if (M == 0) return CF_OK;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    float *P = reinterpret_cast<float *>(w8);
    uint32_t *err = reinterpret_cast<uint32_t *>(w8 + unfused_p_bytes(M, N));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cf_status st = gemm_store_f32(X, W, P, err, M, N, K, s);
    if (st != CF_OK) return st;
    cudaError_t e = cf::launch_row_epilogue(op, P, bias, gamma, beta, static_cast<uint16_t *>(Y), M, int(N), alpha,
                                            eps, rms, static_cast<const uint16_t *>(R), s);
    return e == cudaSuccess ? CF_OK : cuda_fail(e);
}

}  // namespace

extern "C" size_t cf_unfused_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)K;
    if (M < 0 || N <= 0) return cf::kErrBytes;
    return unfused_p_bytes(M, N) + cf::kErrBytes;
}

extern "C" cf_status cf_unfused_gemm_rownorm(const void *X, const void *W, const float *bias, const float *gamma,
                                             const float *beta, void *Y, int64_t M, int64_t N, int64_t K,
                                             float alpha, float eps, cf_activation act, void *workspace,
                                             size_t workspace_bytes, cf_stream_t stream) {
    int op;
    if (act == CF_ACT_NONE) op = 0;
    else if (act == CF_ACT_GELU_TANH) op = 1;
    else return CF_ERR_INVALID_ARG;
    return unfused_common(op, X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, workspace, workspace_bytes, stream);
}

extern "C" cf_status cf_unfused_gemm_rmsnorm(const void *X, const void *W, const float *bias, const float *gamma,
                                             const float *beta, void *Y, int64_t M, int64_t N, int64_t K,
                                             float alpha, float eps, cf_activation act, void *workspace,
                                             size_t workspace_bytes, cf_stream_t stream) {
    int op;
    if (act == CF_ACT_NONE) op = 0;
    else if (act == CF_ACT_GELU_TANH) op = 1;
    else return CF_ERR_INVALID_ARG;
    return unfused_common(op, X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, workspace, workspace_bytes, stream,
                          1);
}

extern "C" cf_status cf_unfused_gemm_residual_norm(const void *X, const void *W, const float *bias, const void *R,
                                                   const float *gamma, const float *beta, void *Y, int64_t M,
                                                   int64_t N, int64_t K, float alpha, float eps, cf_activation act,
                                                   cf_norm norm, void *workspace, size_t workspace_bytes,
                                                   cf_stream_t stream) {
    int op;
    if (act == CF_ACT_NONE) op = 0;
    else if (act == CF_ACT_GELU_TANH) op = 1;
    else return CF_ERR_INVALID_ARG;
    if ((norm != CF_NORM_LAYER && norm != CF_NORM_RMS) || !R) return CF_ERR_INVALID_ARG;
    return unfused_common(op, X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, workspace, workspace_bytes, stream,
                          norm == CF_NORM_RMS ? 1 : 0, R);
}

extern "C" cf_status cf_unfused_gemm_rowsoftmax(const void *X, const void *W, const float *bias, void *Y, int64_t M,
                                                int64_t N, int64_t K, float scale, void *workspace,
                                                size_t workspace_bytes, cf_stream_t stream) {
    return unfused_common(2, X, W, bias, nullptr, nullptr, Y, M, N, K, scale, 0.f, workspace, workspace_bytes,
                          stream);
}
