/*
 * cf.h -- C ABI of libcf: a dense bf16 GEMM fused, in one kernel, with a
 * dependency-rich memory-intensive epilogue (elementwise ops -> row reduction
 * -> broadcast back over the row), plus the GEMM-free stitched
 * reduce -> broadcast subgraph on irregular shapes.  sm_103a (GB300) only.
 *
 * Pages the operations come from (cited by title and section):
 *   [ComFuse]   "ComFuse: Fusing Complex Memory-Intensive Subgraphs with
 *               Compute-Intensive Kernels For Modern GPU Architectures"
 *   [AStitch]   "AStitch: enabling a new multi-dimensional optimization space
 *               for memory-intensive ML training and inference on modern SIMT
 *               architectures"
 *   [sass2mlir] the sass2mlir kernel-fusion page ("Two answers to the same
 *               idle GPU"; section "How we fuse kernels")
 *
 * Conventions for every call
 *   - Pointers marked (device) are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or keeps them.  (host) pointers are
 *     read during the call only.
 *   - Matrices are dense row-major with no padding: X[M,K], W[K,N], Y[M,N].
 *     bf16 is IEEE bfloat16 stored as 16-bit words; fp32 is IEEE binary32.
 *   - Every call is asynchronous and stream-ordered on `stream` (NULL = the
 *     legacy default stream).  The return value reports argument, shape,
 *     alignment, residency and launch errors synchronously; nothing is
 *     launched when it is not CF_OK.
 *   - Errors found on the device (a bounded wait that ran out, an index check)
 *     are recorded in the workspace's error word and reported by
 *     cf_get_device_status().  Kernels never trap: on such an error they
 *     skip the remaining waits, finish, and leave garbage in the output.
 *   - A workspace is caller-owned device memory of at least the size the
 *     matching *_workspace_size() call returns, zeroed once (cf_workspace_init
 *     or cudaMemset) before first use.  Its counters clean themselves at the
 *     end of every launch, so it is reusable by later calls on the same
 *     stream without re-zeroing; it must not be used by two launches that can
 *     run at the same time.  After CF_ERR_DEVICE_TIMEOUT re-zero it.
 *   - Y must not alias X or W (each output element is owned by exactly one
 *     tile: [sass2mlir] "Epilogue fusion - the core technique", ownership
 *     legality).
 */
#ifndef CF_H
#define CF_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CF_API __attribute__((visibility("default")))
#else
#define CF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *cf_stream_t;

typedef enum {
    CF_OK = 0,
    CF_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum      */
    CF_ERR_UNSUPPORTED = 2,        /* shape outside the supported set (below)    */
    CF_ERR_MISALIGNED = 3,         /* pointer not 16-byte aligned                */
    CF_ERR_WORKSPACE_TOO_SMALL = 4,
    CF_ERR_NOT_RESIDENT = 5,       /* the launch cannot keep every CTA that must
                                      meet at an in-kernel barrier resident     */
    CF_ERR_CUDA = 6,               /* a CUDA runtime call failed (see
                                      cf_last_cuda_error)                        */
    CF_ERR_DEVICE_TIMEOUT = 7,     /* device: a bounded wait ran out             */
    CF_ERR_DEVICE_BOUNDS = 8,      /* device: an index check failed              */
    CF_ERR_NO_DEVICE = 9           /* no sm_103 device is current                */
} cf_status;

typedef enum {
    CF_ACT_NONE = 0,
    CF_ACT_GELU_TANH = 1           /* 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))) */
} cf_activation;

/* Human-readable name of a status code (static storage, never NULL). */
CF_API const char *cf_status_string(cf_status status);

/* Library version as 10000*major + 100*minor + patch. */
CF_API int cf_version(void);

/* The cudaError_t of the most recent failing CUDA call made by this thread
 * inside the library (0 if none). */
CF_API int cf_last_cuda_error(void);

/* ------------------------------------------------------------------------ */
/* Tuning knobs.  Every field's zero value means "choose automatically".    */
/* ------------------------------------------------------------------------ */
typedef struct cf_tuning {
    int32_t n_slice;        /* GEMM: columns of one CTA tile (64, 128, 256, 512);
                               B2B: selects the kernel, 128 stream, 256 cluster   */
    int32_t cluster_size;   /* GEMM: CTAs per cluster along the row (1..16)
                               stitched: CTAs per row for the split mapping      */
    int32_t peer_max;       /* inter-CTA aggregation: peer all-to-all when the
                               participating CTA count C_N <= peer_max, else
                               leader-follower ([ComFuse] dual-mode strategy).
                               0 = 8; negative = always leader-follower          */
    int32_t max_clusters;   /* cap on resident clusters of the persistent grid     */
    int32_t stages;         /* GEMM: depth of the shared-memory operand ring;
                               Global BatchNorm: stage buffers of the streaming
                               ring (the CTA's other buffers hold its first
                               stages from the first pass to the second)        */
    int32_t stitch_mapping; /* 0 auto, 1 packed rows, 2 split rows over a cluster  */
    uint32_t timeout_us;    /* bound of every device spin (0 = 200000 us)          */
    int32_t extra_arrivals; /* TEST HOOK: added to the arrival count the global
                               barrier waits for (B2B stream kernel: the
                               per-chunk P-ready barrier); > 0 makes that wait
                               run out (CF_ERR_DEVICE_TIMEOUT) without
                               faulting.  0 in normal use.                        */
    int32_t cluster_m;      /* GEMM: row blocks per cluster (1 or 2); 2 pairs the
                               two row blocks' CTAs into one tcgen05 MMA stream
                               (cta_group::2, M = 256; each CTA stages half of
                               the W tile).  0 = auto                           */
    int32_t disable_pdl;    /* 1 = launch without programmatic dependent
                               launch (by default the kernel's set-up overlaps
                               the previous kernel's tail on the same stream and
                               waits for it before touching memory)            */
    uint64_t *trace;        /* TRACING (fused GEMM): device buffer of
                               grid_ctas * CF_TRACE_SLOTS u64 %globaltimer stamps
                               (ns), or NULL for none.  Per CTA: slots 0..3 =
                               kernel start, set-up done, role loops done, exit;
                               then CF_TRACE_EVENTS slots for each of the CTA's
                               first CF_TRACE_TILES tiles (see cf_trace_event).
                               Slots not reached stay as the caller left them.   */
} cf_tuning;

#define CF_TRACE_TILES 16
#define CF_TRACE_EVENTS 12
#define CF_TRACE_SLOTS (4 + CF_TRACE_TILES * CF_TRACE_EVENTS)

/* Per-tile trace events (slot 4 + tile * CF_TRACE_EVENTS + event). */
typedef enum {
    CF_TR_TMA_FIRST = 0,     /* producer issued the tile's first TMA load      */
    CF_TR_TMA_LAST = 1,      /* producer issued the tile's last TMA load       */
    CF_TR_MMA_ACC_FREE = 2,  /* MMA warp: accumulator buffer free             */
    CF_TR_MMA_FIRST = 3,     /* MMA warp: first operand stage ready            */
    CF_TR_MMA_DONE = 4,      /* MMA warp: last MMA of the tile issued          */
    CF_TR_MMA_WAIT_NS = 5,   /* duration: MMA warp's time waiting for operands */
    CF_TR_EPI_START = 6,     /* epilogue: accumulator ready                    */
    CF_TR_EPI_STATS = 7,     /* epilogue: thread-local statistics done         */
    CF_TR_EPI_CTA = 8,       /* epilogue: CTA statistic done (level 2)         */
    CF_TR_EPI_CLUSTER = 9,   /* epilogue: cluster statistic done (level 3)     */
    CF_TR_EPI_GLOBAL = 10,   /* epilogue: row statistic done (global path)     */
    CF_TR_EPI_STORED = 11    /* epilogue: output stores issued                 */
} cf_trace_event;

/* Per-tile trace events of the back-to-back GEMM kernels (same slot layout;
 * the epilogue's events are stamped by its first thread).  In the stream
 * kernel a "tile" is a 256-column chunk (index = the CTA's chunk count);
 * EPI1_START / EPI2_START mark the chunk's start in the first / second
 * epilogue group, EPI1_LOCAL the softmax exponentials done, EPI1_DONE the
 * chunk's bf16 values written, EPI2_STORED (on a row block's last chunk) the
 * row block's output stored; SENT / RECV are not used. */
typedef enum {
    CF_TRB_TMA_FIRST = 0,    /* producer issued the tile's first load          */
    CF_TRB_ML1_FIRST = 1,    /* MMA warp: first MatMul_1 operand stage ready   */
    CF_TRB_ML1_DONE = 2,     /* MMA warp: MatMul_1 committed                   */
    CF_TRB_EPI1_START = 3,   /* epilogue: P ready in tensor memory             */
    CF_TRB_EPI1_LOCAL = 4,   /* epilogue: CTA-local pass of F done             */
    CF_TRB_EPI1_DONE = 5,    /* epilogue: S written to tensor memory           */
    CF_TRB_ML2_START = 6,    /* MMA warp: S and the O accumulator ready        */
    CF_TRB_ML2_DONE = 7,     /* MMA warp: MatMul_2 committed                   */
    CF_TRB_EPI2_START = 8,   /* epilogue: partial O ready                      */
    CF_TRB_EPI2_SENT = 9,    /* epilogue: partial columns sent to their owners */
    CF_TRB_EPI2_RECV = 10,   /* epilogue: every partial of its columns arrived */
    CF_TRB_EPI2_STORED = 11  /* epilogue: output columns stored                */
} cf_trb_event;

/* Fill *t with the defaults (all zero). */
CF_API void cf_tuning_default(cf_tuning *t);

/* ------------------------------------------------------------------------ */
/* Launch plan (host logic, no GPU needed).                                 */
/* ------------------------------------------------------------------------ */
typedef struct cf_plan {
    int32_t n_slice;        /* tile columns per CTA                                */
    int32_t ctas_per_row;   /* C_total = N / n_slice                               */
    int32_t cluster_size;   /* C_N: CTAs of one cluster along the row              */
    int32_t groups;         /* G = C_total / C_N clusters per row block; G > 1 uses
                               the global partial buffer + in-kernel barrier      */
    int32_t leader_mode;    /* 0 peer all-to-all, 1 leader-follower                */
    int32_t row_blocks;     /* ceil(M / 128)                                       */
    int32_t clusters;       /* clusters of the persistent grid                     */
    int32_t stages;         /* operand ring depth                                  */
    int32_t smem_bytes;     /* dynamic shared memory per CTA                       */
    int32_t cluster_m;      /* C_M: row blocks per cluster; a cluster holds
                               C_M * C_N CTAs; C_M = 2 runs CTA pairs (ranks
                               2i, 2i+1) as one cta_group::2 MMA stream           */
    int32_t staging_buffers;/* bf16 output staging buffers per epilogue warp      */
} cf_plan;

/* Plan a fused GEMM+row-reduce launch for a device with `sm_count` SMs, where
 * max_active_clusters[c] (c = 1..16) is how many clusters of c CTAs (one CTA
 * per SM) can be resident at once (0 = that size cannot launch).  Pure host arithmetic: the
 * same choice the launch calls make after querying the device.
 * Returns CF_UNSUPPORTED for shapes outside the supported set and
 * CF_ERR_NOT_RESIDENT if no residency-valid plan exists. */
CF_API cf_status cf_plan_gemm_fused(int64_t M, int64_t N, int64_t K, int32_t sm_count,
                             const int32_t max_active_clusters[17],
                             const cf_tuning *tuning, cf_plan *plan);

/* The plan the fused GEMM calls would use on the current device for the
 * epilogue `kind` (0 LayerNorm, 1 GELU+LayerNorm, 2 softmax).  Queries the
 * device's residency for every cluster size that could be chosen;
 * max_active_clusters (may be NULL) receives those counts (index = cluster
 * size).  Synchronous, launches nothing. */
CF_API cf_status cf_query_gemm_fused_plan(int64_t M, int64_t N, int64_t K, int32_t kind,
                                          const cf_tuning *tuning, cf_plan *plan,
                                          int32_t max_active_clusters[17]);

/* ------------------------------------------------------------------------ */
/* Workspace                                                                 */
/* ------------------------------------------------------------------------ */

/* Bytes of workspace a fused GEMM call on (M, N, K) may need under any
 * tuning: error word + per-row-block arrival/departure counters + the global
 * partial buffer (one 8-byte statistic per row and cluster group). */
CF_API size_t cf_gemm_fused_workspace_size(int64_t M, int64_t N, int64_t K);

/* Bytes of workspace a stitched call on (rows, cols) needs (error word). */
CF_API size_t cf_stitch_workspace_size(int64_t rows, int64_t cols);

/* Zero `bytes` of the workspace (device) on `stream`. */
CF_API cf_status cf_workspace_init(void *workspace, size_t bytes, cf_stream_t stream);

/* Wait for `stream`, then read and clear the workspace's error word.
 * Returns CF_OK or the first device-side error recorded since the last read;
 * *info (may be NULL) receives where it happened (the row block of a global
 * barrier wait that ran out, or the pipeline wait's role id). */
CF_API cf_status cf_get_device_status(void *workspace, cf_stream_t stream, int32_t *info);

/* ------------------------------------------------------------------------ */
/* Fused GEMM + bias (+GELU) + LayerNorm                                     */
/* ------------------------------------------------------------------------ */
/* Y = LayerNorm_row(act(alpha * X.W + bias)) * gamma + beta
 *
 * [ComFuse] Stage-Stream Execution Model, Fig. 3: stage 1 computes
 * x = alpha*Acc + Bias and the mean reduction; stage 2 reuses x through the
 * bypass path for x - mean; the LayerNorm is the nested "reduce over inputs,
 * normalise using original values" pattern of the Fusion Spec IR (Eq. (10)).
 * Mean and biased variance are taken over the N values of each row (after
 * the activation), eps inside the square root, gamma/beta after normalising.
 *
 *   X     (device) bf16 [M,K] row-major (K contiguous)
 *   W     (device) bf16 [K,N] row-major (N contiguous)
 *   bias  (device) fp32 [N], or NULL for no bias
 *   gamma (device) fp32 [N];  beta (device) fp32 [N]
 *   Y     (device) bf16 [M,N] row-major, written (round to nearest even)
 *   alpha, eps    scalars; act: CF_ACT_NONE or CF_ACT_GELU_TANH
 *   workspace     (device) >= cf_gemm_fused_workspace_size(M,N,K) bytes
 * Accumulation is fp32 in tensor memory; the epilogue is fp32.
 * Supported: M >= 0 (M = 0 is a no-op), K a positive multiple of 64,
 * N a positive multiple of 64 with N / n_slice <= 16 * 64 CTAs per row;
 * X, W, Y, bias, gamma, beta 16-byte aligned.
 * Rows wider than one cluster use the global partial buffer and an in-kernel
 * barrier ([AStitch] "Global" stitching scheme; [sass2mlir] "Grid-barrier
 * synthesis"); this needs every cluster of the persistent grid resident and
 * returns CF_ERR_NOT_RESIDENT otherwise. */
CF_API cf_status cf_gemm_fused_rownorm(const void *X, const void *W, const float *bias,
                                const float *gamma, const float *beta, void *Y,
                                int64_t M, int64_t N, int64_t K, float alpha,
                                float eps, cf_activation act, void *workspace,
                                size_t workspace_bytes, cf_stream_t stream);

CF_API cf_status cf_gemm_fused_rownorm_ex(const void *X, const void *W, const float *bias,
                                   const float *gamma, const float *beta, void *Y,
                                   int64_t M, int64_t N, int64_t K, float alpha,
                                   float eps, cf_activation act, void *workspace,
                                   size_t workspace_bytes, cf_stream_t stream,
                                   const cf_tuning *tuning);

/* Same computation as cf_gemm_fused_rownorm, for callers that cannot
 * allocate device memory: for example a plugin or operator interface that
 * hands its code only the input and output buffers and no allocator, or a
 * runtime that plans every byte of device memory up front and forbids any
 * allocation once it is serving.  The pages have no counterpart to this
 * call; it exists for such callers only.
 *
 * There is no workspace argument and nothing is allocated: no cudaMalloc,
 * cudaFree or allocating library routine is called.  The scratch (error
 * word, barrier counters, global partial buffer) is one fixed device array
 * of 4 MiB inside libcf, which every GPU that loads the library holds until
 * the process exits.  A call needing more scratch than that (256 B + 8 B per
 * 128-row block, rounded up to 256 B, + 1 KiB per 128-row block and cluster
 * group -- rounded up to an even count -- of a row wider than one cluster)
 * returns CF_ERR_WORKSPACE_TOO_SMALL without launching.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array, and each clears its error word and
 *     counters (cudaMemsetAsync on `stream`) before its kernel.  Calls whose
 *     work can overlap on the GPU (different streams, or several host
 *     threads) race on the array and must be serialised by the caller.
 *   - Device-side errors (a bounded wait that ran out: the output is then
 *     garbage) are recorded in the array's error word; read them with
 *     cf_gemm_fused_rownorm_noalloc_status() before the next call, which
 *     clears the word.
 *   - The array's address is cached per device for the life of the process;
 *     after cudaDeviceReset (or anything else that destroys and re-creates
 *     the device's primary context) the cached address is stale, so do not
 *     use this call in a process that resets a device it has used before.
 * Arguments, layouts, supported shapes and error codes are otherwise those
 * of cf_gemm_fused_rownorm with default tuning. */
CF_API cf_status cf_gemm_fused_rownorm_noalloc(const void *X, const void *W, const float *bias,
                                               const float *gamma, const float *beta, void *Y,
                                               int64_t M, int64_t N, int64_t K, float alpha,
                                               float eps, cf_activation act, cf_stream_t stream);

/* The device-side status of cf_gemm_fused_rownorm_noalloc calls on the
 * current device: waits for `stream`, then reads and clears the error word
 * of the library's fixed scratch array (no allocation).  Returns CF_OK or the
 * first device-side error recorded since the last read (or since the last
 * no-allocation call, which clears the word before its kernel); *info (may be
 * NULL) as for cf_get_device_status.  No counterpart in the pages. */
CF_API cf_status cf_gemm_fused_rownorm_noalloc_status(cf_stream_t stream, int32_t *info);

/* ------------------------------------------------------------------------ */
/* Fused GEMM + bias (+ GELU) + RMSNorm                                      */
/* ------------------------------------------------------------------------ */
/* Y = RMSNorm_row(act(alpha * X.W + bias)) * gamma (+ beta), where
 * RMSNorm_row(g) = g / sqrt(mean_row(g^2) + eps) (no mean subtraction).
 *
 * [ComFuse] Fusion Spec IR names RMSNorm among the patterns that become
 * nested stage DAGs: the reduction (mean of the squares) runs over the
 * stage-1 values and the PostOp rescales those values.  The kernel reduces the
 * same per-row (mean, M2) statistics as LayerNorm -- mean(g^2) = M2/N + mean^2
 * -- so every schedule of cf_gemm_fused_rownorm (clusters, the global
 * partial buffer, CTA pairs, wide tiles) applies unchanged.
 * Arguments, layouts, ownership, workspace, supported shapes and errors as for
 * cf_gemm_fused_rownorm, except: beta (device, fp32 [N]) may be NULL (no
 * shift); gamma is required. */
CF_API cf_status cf_gemm_fused_rmsnorm(const void *X, const void *W, const float *bias,
                                       const float *gamma, const float *beta, void *Y,
                                       int64_t M, int64_t N, int64_t K, float alpha,
                                       float eps, cf_activation act, void *workspace,
                                       size_t workspace_bytes, cf_stream_t stream);

CF_API cf_status cf_gemm_fused_rmsnorm_ex(const void *X, const void *W, const float *bias,
                                          const float *gamma, const float *beta, void *Y,
                                          int64_t M, int64_t N, int64_t K, float alpha,
                                          float eps, cf_activation act, void *workspace,
                                          size_t workspace_bytes, cf_stream_t stream,
                                          const cf_tuning *tuning);

/* ------------------------------------------------------------------------ */
/* Fused GEMM + bias (+ GELU) + residual + LayerNorm / RMSNorm               */
/* ------------------------------------------------------------------------ */
typedef enum { CF_NORM_LAYER = 0, CF_NORM_RMS = 1 } cf_norm;

/* Y = Norm(act(alpha * X.W + bias) + R) * gamma (+ beta), Norm = LayerNorm or
 * RMSNorm (`norm`) -- the "add & norm" of a transformer block.
 *
 * [sass2mlir] "Epilogue fusion - the core technique": activation, norm and
 * residual add run on the accumulator in the GEMM's epilogue.  The residual is
 * one more stage-1 node before the row reduction ([ComFuse] Stage-Stream
 * Execution Model); each CTA reads its rows of R once, in pass 1.
 *   R (device) bf16 [M, N] row-major, 16-byte aligned; it may be the same
 *     buffer as Y (every element of R is read by the CTA that later writes
 *     that element of Y, before writing it), but not X or W.
 * Everything else as for cf_gemm_fused_rownorm (CF_NORM_LAYER) or
 * cf_gemm_fused_rmsnorm (CF_NORM_RMS: beta may be NULL). */
CF_API cf_status cf_gemm_fused_residual_norm(const void *X, const void *W, const float *bias,
                                             const void *R, const float *gamma, const float *beta,
                                             void *Y, int64_t M, int64_t N, int64_t K, float alpha,
                                             float eps, cf_activation act, cf_norm norm,
                                             void *workspace, size_t workspace_bytes,
                                             cf_stream_t stream);

CF_API cf_status cf_gemm_fused_residual_norm_ex(const void *X, const void *W, const float *bias,
                                                const void *R, const float *gamma, const float *beta,
                                                void *Y, int64_t M, int64_t N, int64_t K,
                                                float alpha, float eps, cf_activation act,
                                                cf_norm norm, void *workspace,
                                                size_t workspace_bytes, cf_stream_t stream,
                                                const cf_tuning *tuning);

/* ------------------------------------------------------------------------ */
/* Fused GEMM + scaled row softmax                                           */
/* ------------------------------------------------------------------------ */
/* Y = softmax_row(scale * X.W + bias)
 *
 * [ComFuse] Fusion Spec IR: Softmax as a nested reduction (row max, then the
 * sum of exp(z - max)), whose statistics are broadcast back over the row.
 * X, W, Y, workspace as for cf_gemm_fused_rownorm; bias (device) fp32 [N] or
 * NULL.  Same supported shapes. */
CF_API cf_status cf_gemm_fused_rowsoftmax(const void *X, const void *W, const float *bias,
                                   void *Y, int64_t M, int64_t N, int64_t K, float scale,
                                   void *workspace, size_t workspace_bytes,
                                   cf_stream_t stream);

CF_API cf_status cf_gemm_fused_rowsoftmax_ex(const void *X, const void *W, const float *bias,
                                      void *Y, int64_t M, int64_t N, int64_t K,
                                      float scale, void *workspace, size_t workspace_bytes,
                                      cf_stream_t stream, const cf_tuning *tuning);

/* Y = softmax_row(mask(scale * X.W + bias)): the causally masked variant.
 * Column j of row i is kept iff j <= i + offset; masked entries take no part
 * in the row max or sum and are 0 in Y; a row with no kept column is all 0.
 * The pages name the softmax pattern but print no mask: this is the causal
 * mask of attention scores (offset 0 for a square score matrix).  Arguments
 * otherwise as for cf_gemm_fused_rowsoftmax; any offset is accepted. */
CF_API cf_status cf_gemm_fused_rowsoftmax_causal(const void *X, const void *W, const float *bias,
                                                 void *Y, int64_t M, int64_t N, int64_t K,
                                                 float scale, int64_t offset, void *workspace,
                                                 size_t workspace_bytes, cf_stream_t stream);

CF_API cf_status cf_gemm_fused_rowsoftmax_causal_ex(const void *X, const void *W,
                                                    const float *bias, void *Y, int64_t M,
                                                    int64_t N, int64_t K, float scale,
                                                    int64_t offset, void *workspace,
                                                    size_t workspace_bytes, cf_stream_t stream,
                                                    const cf_tuning *tuning);

/* ------------------------------------------------------------------------ */
/* Back-to-back GEMM with the intermediate kept on chip                      */
/* ------------------------------------------------------------------------ */
/* O = bf16( S . W2 ),  S = bf16( F(alpha * X.W1 + b1) )
 *
 * [ComFuse] B2BGEMM, Eqs. 3-7 and Fig. 5, in two kernels; S never reaches
 * global memory in either.
 *  - Cluster kernel (tuning n_slice = 256):
 *    MatMul_1 is partitioned along the intermediate dimension N1 over the
 *    C = N1/256 CTAs of a thread-block cluster (256 columns each); the
 *    epilogue F turns each CTA's P tile into its S tile in tensor memory;
 *    MatMul_2 reads S from there with the CTA's 256-row slice of W2 staged
 *    through the same operand ring as X and W1; the C partial output tiles
 *    are summed across the cluster (in rank order, deterministic) and
 *    written once.  N1 in {256, 512, 1024, 2048}.
 *  - Stream kernel (n_slice = 128; the default): one
 *    CTA per 128-row block; N1 in 256-column chunks through tensor memory,
 *    MatMul_1 of the next chunk running while the epilogue works on the
 *    current one; one O accumulator per row block.  Softmax is evaluated
 *    online (running row max, raised with O rescaled only when a chunk passes
 *    it by 2^8): the bf16 values fed to MatMul_2 are the exponentials against
 *    that running max, and the division by the row sum is applied to the
 *    fp32 O.  LayerNorm in one pass: MatMul_2 takes bf16((z - mu0) gamma1),
 *    mu0 the mean of the row's first 256 columns, while the row (mean, M2)
 *    accumulates; the output is rstd O - rstd (mean - mu0) gamma1^T W2 +
 *    beta1^T W2, the two fp32 rows computed by a small kernel launched just
 *    before on `stream`.  Any N1 that is a multiple of 256.
 *   op   CF_B2B_SOFTMAX: F = row softmax over all N1 columns;
 *        CF_B2B_GELU_TANH: F = GELU(tanh)
 *   X  (device) bf16 [M, K] row-major      W1 (device) bf16 [K, N1] row-major
 *   b1 (device) fp32 [N1] or NULL           W2 (device) bf16 [N1, N2] row-major
 *   O  (device) bf16 [M, N2] row-major, written; must not alias an input
 *   workspace (device) >= cf_b2b_workspace_size() bytes, zeroed once by
 *        cf_workspace_init; holds the device error word (and, for
 *        LayerNorm on the stream kernel, gamma1^T W2, beta1^T W2 and their
 *        partial sums, written by a small kernel launched first on `stream`:
 *        calls sharing a workspace must be ordered on one stream)
 * S is rounded to bf16 before MatMul_2 (the operand precision of the tensor
 * core), as the unfused chain rounds the tensor it stores between the GEMMs.
 * Supported: M >= 0 (0 is a no-op); K > 0 with K % 8 == 0 (a ragged last
 * 64-deep block is zero-filled); N1 % 256 == 0 (cluster kernel: N1 <= 2048);
 * N2 in {64, 128}.
 * All pointers 16-byte aligned (CF_ERR_MISALIGNED).  Asynchronous on
 * `stream`; device-side timeouts are reported by cf_get_device_status. */
typedef enum {
    CF_B2B_SOFTMAX = 0,
    CF_B2B_GELU_TANH = 1,
    CF_B2B_LAYERNORM = 2   /* only through cf_b2b_gemm_layernorm (needs gamma1, beta1) */
} cf_b2b_op;

CF_API size_t cf_b2b_workspace_size(void);

/* The launch the B2B calls would make on the current device: n_slice 256
 * (cluster kernel: cluster_size = C, clusters) or 128 (stream kernel:
 * cluster_size = 1, clusters = CTAs); stages, smem_bytes, row_blocks.  Tuning
 * fields used: n_slice, stages, max_clusters (others ignored).  Synchronous,
 * launches nothing. */
CF_API cf_status cf_query_b2b_plan(int64_t M, int64_t K, int64_t N1, int64_t N2, cf_b2b_op op,
                                   const cf_tuning *tuning, cf_plan *plan);

CF_API cf_status cf_b2b_gemm(const void *X, const void *W1, const float *b1, const void *W2,
                             void *O, int64_t M, int64_t K, int64_t N1, int64_t N2, float alpha,
                             cf_b2b_op op, void *workspace, size_t workspace_bytes,
                             cf_stream_t stream);

/* As cf_b2b_gemm; tuning fields used: n_slice (the kernel), stages,
 * max_clusters (cluster kernel: clusters; stream kernel: CTAs), timeout_us,
 * disable_pdl, trace (per-tile events: cf_trb_event). */
CF_API cf_status cf_b2b_gemm_ex(const void *X, const void *W1, const float *b1, const void *W2,
                                void *O, int64_t M, int64_t K, int64_t N1, int64_t N2,
                                float alpha, cf_b2b_op op, void *workspace,
                                size_t workspace_bytes, cf_stream_t stream,
                                const cf_tuning *tuning);

/* O = bf16( bf16(LayerNorm(alpha * X.W1 + b1) * gamma1 + beta1) . W2 ): the
 * back-to-back GEMM with F = LayerNorm over each row's N1 intermediate
 * values (biased variance, eps inside the square root); the row (mean, M2)
 * is reduced across the cluster like the softmax statistics (stream kernel:
 * over the chunks, applied to the fp32 output as above).  gamma1, beta1
 * (device) fp32 [N1], required; everything else as for cf_b2b_gemm. */
CF_API cf_status cf_b2b_gemm_layernorm(const void *X, const void *W1, const float *b1,
                                       const float *gamma1, const float *beta1, const void *W2,
                                       void *O, int64_t M, int64_t K, int64_t N1, int64_t N2,
                                       float alpha, float eps, void *workspace,
                                       size_t workspace_bytes, cf_stream_t stream);

CF_API cf_status cf_b2b_gemm_layernorm_ex(const void *X, const void *W1, const float *b1,
                                          const float *gamma1, const float *beta1, const void *W2,
                                          void *O, int64_t M, int64_t K, int64_t N1, int64_t N2,
                                          float alpha, float eps, void *workspace,
                                          size_t workspace_bytes, cf_stream_t stream,
                                          const cf_tuning *tuning);

/* ------------------------------------------------------------------------ */
/* Stitched reduce -> broadcast subgraph (no GEMM)                           */
/* ------------------------------------------------------------------------ */
/* out = softmax_row(A*A*A + row_bias[row])
 *
 * [AStitch] "Adaptive thread mapping": very many tiny rows are packed several
 * to a warp (horizontal packing); very few huge rows are split over the CTAs
 * of a cluster (task splitting), the mapping chosen from the actual shape.
 *   A        (device) fp32 [rows, cols] row-major
 *   row_bias (device) fp32 [rows]
 *   out      (device) fp32 [rows, cols] row-major; must not alias A
 *   workspace (device) >= cf_stitch_workspace_size(rows, cols) bytes
 * Supported: rows >= 0, cols >= 0 (either 0 is a no-op), cols <= 262144.
 * 16-byte aligned A/out with cols % 4 == 0 take the 128-bit path; anything
 * else takes the scalar path of the same kernels.
 * Tuning fields used (_ex): stitch_mapping (1 packed, 2 split), cluster_size
 * (CTAs per split row), max_clusters (split: cap on clusters, each then walks
 * several rows with the next row's loads in flight), peer_max, timeout_us,
 * disable_pdl. */
CF_API cf_status cf_stitch_rowreduce_broadcast(const float *A, const float *row_bias, float *out,
                                        int64_t rows, int64_t cols, void *workspace,
                                        size_t workspace_bytes, cf_stream_t stream);

CF_API cf_status cf_stitch_rowreduce_broadcast_ex(const float *A, const float *row_bias,
                                           float *out, int64_t rows, int64_t cols,
                                           void *workspace, size_t workspace_bytes,
                                           cf_stream_t stream, const cf_tuning *tuning);

/* ------------------------------------------------------------------------ */
/* Stitched power -> broadcast -> add -> row softmax                          */
/* ------------------------------------------------------------------------ */
/* out[i, j] = softmax_j(A[i, j] + w[j]^p): an expensive element-wise power of a
 * column vector, broadcast to every row, added, then the row softmax.
 *
 * [AStitch] "What people did before" names power -> broadcast -> add as the
 * pattern register-only fusion recomputes once per consumer element;
 * "Four stitching schemes" gives it the Regional scheme: every CTA computes the
 * powers of the columns it touches once, into shared memory, and every row it
 * handles reads them there.  The row softmax and its thread mapping (packed
 * rows up to 128 columns, cluster-split wider rows) are those of
 * cf_stitch_rowreduce_broadcast.
 *   A   (device) fp32 [rows, cols] row-major     w (device) fp32 [cols], > 0
 *   p   exponent (host scalar); w^p is the real power 2^(p log2 w): a w <= 0
 *       gives NaN or 0 in its column, as the power function has no real value
 *       or zero there
 *   out (device) fp32 [rows, cols]; must not alias A or w
 * Pointers 4-byte aligned (16-byte aligned A/out with cols % 4 == 0 take the
 * 128-bit path); cols <= 262144 (else CF_ERR_UNSUPPORTED); workspace and
 * device-side errors as for cf_stitch_rowreduce_broadcast. */
CF_API cf_status cf_stitch_powadd_softmax(const float *A, const float *w, float p, float *out, int64_t rows,
                                          int64_t cols, void *workspace, size_t workspace_bytes,
                                          cf_stream_t stream);

CF_API cf_status cf_stitch_powadd_softmax_ex(const float *A, const float *w, float p, float *out, int64_t rows,
                                             int64_t cols, void *workspace, size_t workspace_bytes,
                                             cf_stream_t stream, const cf_tuning *tuning);

/* out = LayerNorm(A + R) * gamma + beta over each row
 *
 * [AStitch] "Four stitching schemes": an elementwise producer (A + R), two
 * row reductions (the mean, then the variance around it) and their
 * broadcast, with column parameters shared by every row, in one kernel; the
 * thread mapping is that of cf_stitch_rowreduce_broadcast (rows of up to 128
 * columns packed several to a warp, wider rows split over the CTAs of a
 * cluster with one DSMEM exchange of (mean, M2) per row).
 *   A, R  (device) fp32 [rows, cols] row-major; R may be NULL (out = LN(A))
 *   gamma, beta (device) fp32 [cols]
 *   out   (device) fp32 [rows, cols]; may alias A (each element is read before
 *         it is written, by the thread that writes it)
 *   variance biased (divide by cols), eps inside the square root
 *   workspace >= cf_stitch_workspace_size(rows, cols) bytes
 * Supported: rows, cols >= 0 (0 is a no-op), cols <= 262144; 4-byte aligned
 * pointers (16-byte aligned with cols % 4 == 0 takes the 128-bit path).
 * Tuning fields used: stitch_mapping (1 packed, 2 split), cluster_size,
 * timeout_us, disable_pdl. */
CF_API cf_status cf_stitch_add_layernorm(const float *A, const float *R, const float *gamma,
                                         const float *beta, float *out, int64_t rows, int64_t cols,
                                         float eps, void *workspace, size_t workspace_bytes,
                                         cf_stream_t stream);

CF_API cf_status cf_stitch_add_layernorm_ex(const float *A, const float *R, const float *gamma,
                                            const float *beta, float *out, int64_t rows,
                                            int64_t cols, float eps, void *workspace,
                                            size_t workspace_bytes, cf_stream_t stream,
                                            const cf_tuning *tuning);

/* out = (A - mean_col) / sqrt(var_col + eps) * gamma[col] + beta[col]
 * with the batch statistics of each column (mean and biased variance over all
 * rows), as BatchNorm computes them in training.
 *
 * [AStitch] "Four stitching schemes": the column statistic is a one-to-many
 * dependency over every row.  Regional (rows <= 256): one CTA holds all rows
 * of a 128-column strip in registers and combines its warps' partials in
 * shared memory -- one HBM pass.  Global (more rows): one resident wave of
 * CTAs (vertical packing) reduces contiguous row ranges, writes column
 * partials to the workspace and meets at an in-kernel grid barrier; every
 * CTA folds all partials in one fixed order, then normalises its rows,
 * re-reading them from L2 where they still are.  The launch is refused
 * (CF_ERR_NOT_RESIDENT) if the wave cannot be resident.
 *   A     (device) fp32 [rows, cols] row-major
 *   gamma, beta (device) fp32 [cols]
 *   out   (device) fp32 [rows, cols]; must not alias A
 *   mean_out, var_out (device) fp32 [cols] or NULL: the batch statistics
 *   workspace (device) >= cf_stitch_batchnorm_workspace_size(rows, cols)
 *         bytes, 16-byte aligned, zeroed once by cf_workspace_init; the grid
 *         barrier's counters reset themselves at the end of each launch (after
 *         a device-side error, zero the workspace again)
 * Supported: rows, cols >= 0 (0 is a no-op); 4-byte aligned pointers.
 * Tuning fields used: stitch_mapping (3 Regional, 4 Global), max_clusters
 * (cap on the Global grid), stages (Global with 16-byte aligned rows: the
 * stage buffers of each CTA's streaming ring, the others holding its first
 * stages between the passes; 0 = 128 KB of ring), timeout_us, disable_pdl,
 * extra_arrivals (TEST HOOK: > 0 makes the grid barrier wait run out). */
CF_API size_t cf_stitch_batchnorm_workspace_size(int64_t rows, int64_t cols);

CF_API cf_status cf_stitch_batchnorm(const float *A, const float *gamma, const float *beta,
                                     float *out, float *mean_out, float *var_out, int64_t rows,
                                     int64_t cols, float eps, void *workspace,
                                     size_t workspace_bytes, cf_stream_t stream);

CF_API cf_status cf_stitch_batchnorm_ex(const float *A, const float *gamma, const float *beta,
                                        float *out, float *mean_out, float *var_out, int64_t rows,
                                        int64_t cols, float eps, void *workspace,
                                        size_t workspace_bytes, cf_stream_t stream,
                                        const cf_tuning *tuning);

/* The mapping (3 Regional, 4 Global) and grid size the BatchNorm call would
 * use on the current device.  Synchronous, launches nothing. */
CF_API cf_status cf_query_stitch_batchnorm_plan(int64_t rows, int64_t cols, const cf_tuning *tuning,
                                                int32_t *mapping, int32_t *grid);

/* ------------------------------------------------------------------------ */
/* The unfused two-kernel composition (measured baseline)                    */
/* ------------------------------------------------------------------------ */
/* The same computations as cf_gemm_fused_rownorm / cf_gemm_fused_rowsoftmax,
 * scheduled the way fusion avoids: kernel 1 writes P = X.W as fp32 [M,N] into
 * the workspace (the intermediate that [ComFuse] Stage-Stream Execution Model
 * keeps out of GMEM), kernel 2 reads it back and applies bias (GELU) and the
 * row reduction + broadcast.  For measuring what fusion saves; not a
 * fallback.  Arguments as for the fused calls; the workspace (device,
 * >= cf_unfused_workspace_size bytes, 16-byte aligned) holds P and an error
 * word.  Supported: N a multiple of 64 up to 16384, K a multiple of 64. */
CF_API size_t cf_unfused_workspace_size(int64_t M, int64_t N, int64_t K);

CF_API cf_status cf_unfused_gemm_rownorm(const void *X, const void *W, const float *bias,
                                         const float *gamma, const float *beta, void *Y,
                                         int64_t M, int64_t N, int64_t K, float alpha, float eps,
                                         cf_activation act, void *workspace,
                                         size_t workspace_bytes, cf_stream_t stream);

/* The unfused composition of cf_gemm_fused_rmsnorm (beta may be NULL). */
CF_API cf_status cf_unfused_gemm_rmsnorm(const void *X, const void *W, const float *bias,
                                         const float *gamma, const float *beta, void *Y,
                                         int64_t M, int64_t N, int64_t K, float alpha, float eps,
                                         cf_activation act, void *workspace,
                                         size_t workspace_bytes, cf_stream_t stream);

/* The unfused composition of cf_gemm_fused_residual_norm. */
CF_API cf_status cf_unfused_gemm_residual_norm(const void *X, const void *W, const float *bias,
                                               const void *R, const float *gamma, const float *beta,
                                               void *Y, int64_t M, int64_t N, int64_t K, float alpha,
                                               float eps, cf_activation act, cf_norm norm,
                                               void *workspace, size_t workspace_bytes,
                                               cf_stream_t stream);

CF_API cf_status cf_unfused_gemm_rowsoftmax(const void *X, const void *W, const float *bias,
                                            void *Y, int64_t M, int64_t N, int64_t K, float scale,
                                            void *workspace, size_t workspace_bytes,
                                            cf_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CF_H */
