// umma.cuh -- descriptors of the 5th-generation tensor core MMA (tcgen05.mma,
// kind::f16) shared by the fused kernels: the shared-memory matrix descriptor
// for 128-byte swizzled operand tiles and the instruction descriptor.
#pragma once

#include <cstdint>

namespace cf {

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;  // descriptor version for tcgen05
    d |= uint64_t(2) << 61;  // SWIZZLE_128B
    return d;
}

// instruction descriptor: kind::f16, A = B = bf16, D = fp32, A K-major,
// B MN-major (W is [K,N] with N contiguous), M = m (128, or 256 for a CTA pair), N = n
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) | (uint32_t(n >> 3) << 17) |
           (uint32_t(m >> 4) << 24);
}


}  // namespace cf
