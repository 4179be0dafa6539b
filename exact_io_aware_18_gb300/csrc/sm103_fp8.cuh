// sm103_fp8.cuh - 8-bit float tensor-core primitives for sm_103a (inline PTX).
#pragma once

#include <cstdint>

namespace fa {

// Instruction descriptor, kind::f8f6f4: E4M3 A and B (format code 0), FP32
// accumulator, dense, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) |                              // D: f32
           (0u << 7) |                              // A: e4m3
           (0u << 10) |                             // B: e4m3
           (static_cast<uint32_t>(N >> 3) << 17) |  // N / 8
           (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// D(tmem) (+)= A(smem) * B(smem), kind::f8f6f4, one CTA: 32 elements (32
// bytes) of K per instruction.
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

}  // namespace fa
