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

// Shared-memory matrix descriptor for a 64-byte-swizzled K-major operand:
// rows of 64 bytes (64 E4M3 codes), 512-byte atoms of 8 rows whose 16-byte
// chunks are XOR-ed with the address bits above them, every atom 512-byte
// aligned.  sbo is the byte stride between 8-row groups (512 for a dense
// tile); the leading offset is not used.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr, uint32_t sbo_bytes) {
    const uint32_t lo = ((saddr & 0x3FFFFu) >> 4) | (1u << 16);  // leading offset (unused)
    const uint32_t hi = ((sbo_bytes >> 4) & 0x3FFFu) |
                        (1u << 14) |  // descriptor version for tcgen05 (bit 46)
                        (4u << 29);   // 64-byte swizzle (bits 61-63)
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

}  // namespace fa
