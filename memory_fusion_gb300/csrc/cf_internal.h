// cf_internal.h -- launchers shared between the C-ABI layer (cf_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace cf {

// Workspace layout (device, caller-owned, zeroed once):
//   [0, 256)                 error word: u32 status, u32 info, rest reserved
//   [256, 256 + 8*RB pad)    per-row-block counters: arrive[RB], depart[RB]
//   [...]                    global partials: [RB][128][G rounded up to even] float2
constexpr size_t kErrBytes = 256;
constexpr int kBlockM = 128;  // rows of one GEMM tile (tcgen05 M = 128, one row per TMEM lane)

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int max_smem_optin = 0;
};

// Returns the current device's info (cached per device).  false if none.
bool current_device_info(DeviceInfo *out);

// --------------------------------------------------------------------------
// stitched kernels (stitch.cu)
// --------------------------------------------------------------------------
struct StitchPlan {
    int mapping = 0;      // 1 packed, 2 split
    int lpr = 0;          // packed: lanes per row (1..32, power of two)
    int cluster = 0;      // split: CTAs per row
    int per_thread = 0;   // split: float4 groups per thread (1..16, power of two)
    int leader = 0;       // split: leader-follower aggregation
    bool vec = false;     // 128-bit path
    bool pdl = true;      // programmatic dependent launch
    int grid = 0;         // CTAs
    unsigned long long timeout_ns = 200000000ull;  // bound of every wait (split mapping)
};

// y = A^3 + bias[row] (w == null), or y = A + w[col]^pexp (w != null, w > 0),
// then the row softmax
cudaError_t launch_stitch(const StitchPlan &p, const float *A, const float *bias, float *out, int64_t rows,
                          int64_t cols, uint32_t *err, cudaStream_t stream, const float *w = nullptr,
                          float pexp = 0.f);

int stitch_packed_blocks_per_sm(int lpr, bool vec);

// --------------------------------------------------------------------------
// stitched normalisation subgraphs (stitch_norm.cu)
// --------------------------------------------------------------------------
// add + LayerNorm over rows: mapping 1 packed (lpr), 2 split (cluster, per_thread)
cudaError_t launch_add_layernorm(const StitchPlan &p, const float *A, const float *R, const float *gamma,
                                 const float *beta, float *out, int64_t rows, int64_t cols, float eps, uint32_t *err,
                                 cudaStream_t stream);
int addln_packed_blocks_per_sm(int lpr, bool vec);

// BatchNorm over columns: mapping 3 Regional (one CTA per 128-column strip
// holding all rows, rpt rows per warp), 4 Global (strips x chunks resident
// CTAs of 1024 threads, in-kernel grid barrier)
struct BnPlan {
    int mapping = 0;
    int rpt = 0;          // Regional: rows per warp held in registers (1..32, power of two)
    int lpr = 0;          // Global: 4-column groups per strip (1..32, power of two)
    int strips = 0;       // Global: column strips
    int grid = 0;
    bool vec = false;
    bool pdl = true;
    int extra_arrivals = 0;
    bool tma = false;     // Global: stream the rows through shared memory by TMA
    int64_t rows_per_chunk = 0;  // Global + TMA: a multiple of the stage height
    unsigned long long timeout_ns = 200000000ull;
};
cudaError_t launch_batchnorm(const BnPlan &p, const float *A, const float *gamma, const float *beta, float *out,
                             float *mean_out, float *var_out, int64_t rows, int64_t cols, float eps, uint32_t *err,
                             uint32_t *counters, float2 *partials, cudaStream_t stream);
int bn_global_blocks_per_sm(int lpr, bool vec);

// Global BatchNorm streamed through shared memory by TMA (cols % 4 == 0,
// 16-byte aligned A and out): one producer warp, eight compute warps
struct BnTmaArgs {
    CUtensorMap tmap_a;    // A [rows, cols] fp32, box (4*lpr) x br, no swizzle
    const float *gamma, *beta;
    float *mean_out, *var_out;
    uint32_t *err, *counters;
    float2 *partials;      // [grid][4*lpr]
    int64_t rows;
    int cols, strips, rows_per_chunk, extra_arrivals;
    float eps;
    unsigned long long timeout_ns;
    unsigned long long *trace;  // optional: per CTA slots 0..3 = start, pass 1 done, barrier passed, pass 2 done
    const float *A;        // flat (cols == 4*lpr): stages load as untiled bulk copies
    float *out;            // [rows, cols], written from registers
    int flat;
    int ring, res;  // stage buffers streaming, and holding the first stages resident
};
cudaError_t launch_batchnorm_tma(int lpr, const BnTmaArgs &a, int grid, bool pdl, cudaStream_t stream);
int bn_tma_blocks_per_sm(int lpr);
int bn_tma_box_rows(int lpr);   // rows of one stage for a strip of 4*lpr columns
// split the CTA's stage buffers into a streaming ring (`stages` of them, 0 =
// default) and resident stages
void bn_tma_buffers(int lpr, int stages, int *ring, int *res);
// row slots a thread takes per iteration in the packed stitched kernels (the
// softmax and add + LayerNorm ones): one, so that a thread needs few
// registers and the SM holds 2048 threads; at four, add + LayerNorm over
// 750000x32 took 55.9 us instead of 44.5 (73 registers, 768 threads an SM)
constexpr int kPackedUnroll = 1;
constexpr int kBnRegionalMaxRows = 256;   // 8 warps x 32 rows in registers
constexpr int kBnMaxGlobalCtas = 1024;    // bound of the partial buffer

// --------------------------------------------------------------------------
// row epilogue kernel of the unfused baseline (rowkernel.cu):
//   op 0 LN, 1 GELU+LN, 2 softmax over fp32 rows of P -> bf16 Y
// --------------------------------------------------------------------------
cudaError_t launch_row_epilogue(int op, const float *P, const float *bias, const float *gamma, const float *beta,
                                uint16_t *Y, int64_t M, int N, float alpha, float eps, int rms, const uint16_t *R,
                                cudaStream_t stream);

// --------------------------------------------------------------------------
// fused GEMM kernels (gemm_fused.cu)
// --------------------------------------------------------------------------
enum EpiKind : int {
    EPI_LN = 0,        // alpha*acc + bias -> LayerNorm -> bf16
    EPI_GELU_LN = 1,   // alpha*acc + bias -> GELU(tanh) -> LayerNorm -> bf16
    EPI_SOFTMAX = 2,   // scale*acc + bias -> softmax -> bf16
    EPI_STORE_F32 = 3, // raw fp32 accumulator to P [M,N] (the unfused baseline's GEMM)
    EPI_SOFTMAX_MASK = 4,  // EPI_SOFTMAX over the causally masked row (keep col <= row + offset)
};

struct GemmArgs {
    CUtensorMap tmap_x;   // X [M,K] bf16, box 64(K) x (128/C_N)(M), 128B swizzle
    CUtensorMap tmap_w;   // W [K,N] bf16, box 64(N) x 64(K), 128B swizzle
    CUtensorMap tmap_y;   // Y [M,N] bf16, box 32(N) x 32(M), 64B swizzle (stores);
                          // EPI_STORE_F32: P [M,N] fp32, box 16(N) x 32(M)
    const float *bias;    // [N] or null
    const float *gamma;   // [N] (LN, RMSNorm)
    const float *beta;    // [N] (LN; RMSNorm: or null)
    uint16_t *y;          // [M,N] bf16
    uint32_t *err;        // workspace error word
    uint32_t *counters;   // [2*RB]: arrive, depart
    float2 *partials;     // [RB][Gp][128]
    int M, N, K;
    float alpha;          // LN: multiplies acc; softmax: scale
    float eps;
    int n_slice;          // columns of one tile
    int cluster;          // C_N: CTAs of one row group (along N)
    int cluster_m;        // C_M: row blocks per cluster; 2 = CTA pairs sharing one
                          // cta_group::2 MMA stream (M = 256, W split between the pair)
    int stg_bufs;         // output staging buffers per epilogue warp (1 or 2)
    int groups;           // G
    int leader;           // leader-follower aggregation in the row group
    int row_blocks;       // RB = ceil(M / 128)
    int row_blocks_alloc; // RB rounded up to a multiple of C_M (counter / partial rows)
    int super_blocks;     // RB_alloc / C_M
    int extra_arrivals;   // test hook
    int rms;              // LN kinds: normalise by sqrt(mean(g^2) + eps), no centring (RMSNorm)
    const uint16_t *resid;  // LN kinds: bf16 [M,N] residual added after the activation, or null
    long long mask_offset;  // EPI_SOFTMAX_MASK: column j of row i is kept iff j <= i + mask_offset
    unsigned long long timeout_ns;
    unsigned long long *trace;  // optional %globaltimer stamps, CF_TRACE_SLOTS per CTA
};

// dynamic shared memory of one CTA for a ring of `stages`, a row group of
// `cluster` CTAs, the CTA-pair MMA mode or not, leader-follower or peer exchange
int gemm_fused_smem_bytes(int stages, int cluster, int n_slice, bool pair, bool leader, int stg_bufs);

// Query max co-resident clusters of `cluster` CTAs (total) for the fused
// kernel of `kind` and mode with `smem` dynamic shared memory (0 if it cannot
// launch).
int gemm_fused_max_active_clusters(int kind, bool pair, int cluster, int smem);

// pdl: allow programmatic dependent launch (the kernel waits on griddepcontrol
// before touching global memory)
cudaError_t launch_gemm_fused(int kind, const GemmArgs &a, int clusters, int stages, int smem, bool pdl,
                              cudaStream_t stream);

// --------------------------------------------------------------------------
// back-to-back GEMM (b2b.cu): O = F(alpha * X.W1 + b1) . W2, F = softmax / GELU
// --------------------------------------------------------------------------
struct B2bArgs {
    CUtensorMap tmap_x;   // X [M,K] bf16, box 64(K) x 128(M), 128B swizzle
    CUtensorMap tmap_w1;  // W1 [K,N1] bf16 as {64, K, N1/64}, box {64, 64, 4}
    CUtensorMap tmap_w2;  // W2 [N1,N2] bf16 as {64, N1, N2/64}, box {64, 64, N2/64}
    CUtensorMap tmap_o;   // stream kernel: O [M,N2] bf16, box 32 x 32, 64B swizzle (TMA stores)
    const float *b1;      // [N1] or null
    const float *gamma1;  // LayerNorm F: [N1]
    const float *beta1;   // LayerNorm F: [N1]
    float eps;            // LayerNorm F
    uint16_t *out;        // O [M,N2] bf16
    uint32_t *err;        // workspace error word
    int M, K, N1, N2;
    int cluster;          // C = N1 / 256 CTAs per row block
    float alpha;
    unsigned long long timeout_ns;
    unsigned long long *trace;  // optional %globaltimer stamps, CF_TRACE_SLOTS per CTA
    int extra_arrivals;   // test hook (stream kernel): added to the per-chunk P-ready count
    const float *fold;    // stream kernel, LayerNorm F: c1 = gamma1^T W2, c0 = beta1^T W2 (fp32 [2][N2])
};

int b2b_smem_bytes(int stages, int cluster, int n2, int op);
int b2b_max_active_clusters(int op, int cluster, int n2, int smem);
cudaError_t launch_b2b(int op, const B2bArgs &a, int clusters, int stages, int smem, bool pdl, cudaStream_t stream);
// one CTA per 128-row block, N1 streamed in 256-column chunks (softmax, GELU, LayerNorm);
// tmap_w1 box {64, 64, 4}, tmap_w2 box {64, 128, N2/64}
int b2b_stream_stages(int op, int K);  // ring depth, fixed per epilogue and mode (X resident or streamed)
int b2b_stream_smem_bytes(int op, int K);
cudaError_t launch_b2b_stream(int op, const B2bArgs &a, int ctas, int smem, bool pdl, cudaStream_t stream);
// The stream kernel's LayerNorm output terms c1 = gamma1^T W2 and c0 = beta1^T W2
// (fp32, fixed summation order), computed by a small kernel launched before it.
// Workspace: the error word, c [2][128] fp32, two counters, the partial sums.
constexpr int kB2bFoldSplits = 32;
constexpr size_t kB2bFoldOff = kErrBytes;
constexpr size_t kB2bFoldCountersOff = kB2bFoldOff + 2 * 128 * sizeof(float);
constexpr size_t kB2bFoldPartialsOff = kB2bFoldCountersOff + 256;
constexpr size_t kB2bWorkspaceBytes = kB2bFoldPartialsOff + size_t(kB2bFoldSplits) * 2 * 128 * sizeof(float);
cudaError_t launch_b2b_ln_fold(const void *W2, const float *gamma1, const float *beta1, int N1, int N2,
                               unsigned char *ws, bool pdl, cudaStream_t stream);

}  // namespace cf
