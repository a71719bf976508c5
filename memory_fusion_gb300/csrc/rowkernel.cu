// rowkernel.cu -- the second kernel of the unfused two-kernel composition used
// as a measured baseline next to the fused kernel: it reads the fp32 GEMM
// result P [M, N] back from global memory and applies the memory-intensive
// subgraph row by row:
//     op 0 (LN):       y = LayerNorm(alpha*P + bias) * gamma + beta
//     op 1 (GELU_LN):  y = LayerNorm(GELU_tanh(alpha*P + bias)) * gamma + beta
//     op 2 (SOFTMAX):  y = softmax(alpha*P + bias)
// (ops 0 and 1 with `rms`: RMSNorm, y = g / sqrt(mean(g^2) + eps) * gamma + beta;
//  with a residual R [M,N] bf16, g = act(alpha*P + bias) + R)
// This is the materialised-intermediate schedule the fusion removes ([ComFuse]
// Stage-Stream Execution Model: an edge that would otherwise be a buffer in
// GMEM); it exists so the cost of that buffer can be measured, not as a
// fallback.  One CTA per row: each thread keeps VPT values of the row in
// registers; the reduction is warp butterfly -> shared memory -> CTA.
#include <cuda_runtime.h>

#include <cstdint>

#include "cf_internal.h"
#include "ptx.cuh"
#include "rowstats.cuh"

namespace cf {
namespace {

constexpr int kRowThreads = 256;

// (count, mean, M2) of a thread's values, combined with Chan's update
struct Stat3 {
    float n, mean, m2;
};

__device__ __forceinline__ Stat3 combine3(Stat3 a, Stat3 b) {
    const float n = a.n + b.n;
    if (n == 0.f) return a;
    const float d = b.mean - a.mean;
    const float f = b.n / n;
    return Stat3{n, a.mean + d * f, a.m2 + b.m2 + d * d * a.n * f};
}

template <int OP, int VPT>
__global__ void __launch_bounds__(kRowThreads) row_epilogue_kernel(const float *__restrict__ P,
                                                                   const float *__restrict__ bias,
                                                                   const float *__restrict__ gamma,
                                                                   const float *__restrict__ beta,
                                                                   uint16_t *__restrict__ Y, int64_t M, int N,
                                                                   float alpha, float eps, int rms,
                                                                   const uint16_t *__restrict__ R) {
    constexpr int G4 = VPT / 4;  // float4 groups per thread; group j holds columns (j*256 + t)*4 ..
    __shared__ float4 red[kRowThreads / 32];
    __shared__ float2 fin;
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    ptx::griddep_wait();
    for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
        const float *prow = P + r * N;
        float x[VPT];
#pragma unroll
        for (int j = 0; j < G4; ++j) {
            const int c = (j * kRowThreads + t) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f), b = v;
            if (c < N) {
                v = __ldcs(reinterpret_cast<const float4 *>(prow + c));
                if (bias) b = __ldg(reinterpret_cast<const float4 *>(bias + c));
            }
            x[4 * j + 0] = fmaf(alpha, v.x, b.x);
            x[4 * j + 1] = fmaf(alpha, v.y, b.y);
            x[4 * j + 2] = fmaf(alpha, v.z, b.z);
            x[4 * j + 3] = fmaf(alpha, v.w, b.w);
        }
        float2 stat;
        if constexpr (OP == 2) {
            float m = neg_inf();
#pragma unroll
            for (int j = 0; j < G4; ++j)
                if ((j * kRowThreads + t) * 4 < N)
#pragma unroll
                    for (int k = 0; k < 4; ++k) m = fmaxf(m, x[4 * j + k]);
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < G4; ++j) {
                const bool ok = (j * kRowThreads + t) * 4 < N;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float e = ok ? ptx::ex2_approx((x[4 * j + k] - m) * kLog2e) : 0.f;
                    x[4 * j + k] = e;
                    s += e;
                }
            }
            MaxSum p = warp_maxsum<32>(MaxSum{m, s});
            if (lane == 0) red[warp] = make_float4(p.m, p.s, 0.f, 0.f);
            __syncthreads();
            if (warp == 0) {
                MaxSum q = lane < kRowThreads / 32 ? MaxSum{red[lane].x, red[lane].y} : MaxSum{neg_inf(), 0.f};
                q = warp_maxsum<kRowThreads / 32>(q);
                if (lane == 0) fin = make_float2(q.m, q.s);
            }
            __syncthreads();
            const float f = ptx::ex2_approx((m - fin.x) * kLog2e) / fin.y;
#pragma unroll
            for (int k = 0; k < VPT; ++k) x[k] *= f;
            stat = fin;
        } else {
            Stat3 st{0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < G4; ++j) {
                if ((j * kRowThreads + t) * 4 >= N) continue;
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if constexpr (OP == 1) x[4 * j + k] = gelu_tanh_dev(x[4 * j + k]);
                    if (R) {
                        const uint32_t w = reinterpret_cast<const uint32_t *>(R + r * N + (j * kRowThreads + t) * 4)[k >> 1];
                        x[4 * j + k] += __uint_as_float((k & 1) ? (w & 0xFFFF0000u) : (w << 16));
                    }
                    s += x[4 * j + k];
                }
                const float mu = 0.25f * s;
                float m2 = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) m2 = fmaf(x[4 * j + k] - mu, x[4 * j + k] - mu, m2);
                st = combine3(st, Stat3{4.f, mu, m2});
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                Stat3 o{__shfl_xor_sync(0xffffffffu, st.n, off), __shfl_xor_sync(0xffffffffu, st.mean, off),
                        __shfl_xor_sync(0xffffffffu, st.m2, off)};
                st = (lane & off) ? combine3(o, st) : combine3(st, o);
            }
            if (lane == 0) red[warp] = make_float4(st.n, st.mean, st.m2, 0.f);
            __syncthreads();
            if (t == 0) {
                Stat3 a{red[0].x, red[0].y, red[0].z};
                for (int w = 1; w < kRowThreads / 32; ++w) a = combine3(a, Stat3{red[w].x, red[w].y, red[w].z});
                const float var = a.m2 / float(N);
                fin = rms ? make_float2(0.f, rsqrtf(fmaf(a.mean, a.mean, var) + eps))
                          : make_float2(a.mean, rsqrtf(var + eps));
            }
            __syncthreads();
            stat = fin;
        }
        uint16_t *yrow = Y + r * N;
#pragma unroll
        for (int j = 0; j < G4; ++j) {
            const int c = (j * kRowThreads + t) * 4;
            if (c >= N) continue;
            float y0 = x[4 * j], y1 = x[4 * j + 1], y2 = x[4 * j + 2], y3 = x[4 * j + 3];
            if constexpr (OP != 2) {
                const float4 g = __ldg(reinterpret_cast<const float4 *>(gamma + c));
                const float4 b = beta ? __ldg(reinterpret_cast<const float4 *>(beta + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
                y0 = fmaf((y0 - stat.x) * stat.y, g.x, b.x);
                y1 = fmaf((y1 - stat.x) * stat.y, g.y, b.y);
                y2 = fmaf((y2 - stat.x) * stat.y, g.z, b.z);
                y3 = fmaf((y3 - stat.x) * stat.y, g.w, b.w);
            }
            uint2 w;
            w.x = ptx::pack_bf16x2(y0, y1);
            w.y = ptx::pack_bf16x2(y2, y3);
            *reinterpret_cast<uint2 *>(yrow + c) = w;
        }
        __syncthreads();  // red / fin are reused by the next row
    }
    ptx::griddep_launch_dependents();
}

template <int OP>
void *row_fn(int vpt) {
    switch (vpt) {
        case 4: return reinterpret_cast<void *>(&row_epilogue_kernel<OP, 4>);
        case 8: return reinterpret_cast<void *>(&row_epilogue_kernel<OP, 8>);
        case 16: return reinterpret_cast<void *>(&row_epilogue_kernel<OP, 16>);
        case 32: return reinterpret_cast<void *>(&row_epilogue_kernel<OP, 32>);
        case 64: return reinterpret_cast<void *>(&row_epilogue_kernel<OP, 64>);
        default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_row_epilogue(int op, const float *P, const float *bias, const float *gamma, const float *beta,
                                uint16_t *Y, int64_t M, int N, float alpha, float eps, int rms, const uint16_t *R,
                                cudaStream_t stream) {
    int vpt = 4;
    while (vpt * kRowThreads < N) vpt *= 2;
    if (vpt > 64) return cudaErrorInvalidValue;
    void *fn = op == 0 ? row_fn<0>(vpt) : op == 1 ? row_fn<1>(vpt) : op == 2 ? row_fn<2>(vpt) : nullptr;
    if (!fn) return cudaErrorInvalidValue;
    const int64_t grid = M < 65536 ? M : 65536;
    void *args[] = {(void *)&P, (void *)&bias, (void *)&gamma, (void *)&beta, (void *)&Y, (void *)&M, (void *)&N,
                    (void *)&alpha, (void *)&eps, (void *)&rms, (void *)&R};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kRowThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace cf
