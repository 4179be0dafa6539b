// fp8_quant_sm103.cu - incoherent processing and block quantisation of Q or K
// for the FP8 forward (memory-bound).
//
// "FlashAttention scaling, multi-GPU training and weight quantization"
// (section 1, FlashAttention-3, FP8 low-precision support): before Q and K go
// to 8-bit floats they are multiplied by a random orthogonal matrix, which
// spreads outlier channels over all channels, and every small tile is scaled
// on its own.  Here the matrix is R = diag(s) H / sqrt(d), H the Sylvester
// Hadamard matrix and s a vector of random signs, so x R is a fast
// Walsh-Hadamard transform of x with its signs flipped; a tile is 128 rows of
// one head.  Per tile, with amax the largest |x R|:
//     code  = E4M3(x R * (448 / amax))  (round to nearest even, saturating)
//     scale = amax / 448                 (dequantisation: x R ~ code * scale)
// and an all-zero tile gets codes 0 and scale 1.  Scores are unchanged by the
// rotation, Q R (K R)^T = Q K^T, so the FP8 forward applies no inverse.
//
// The codes must come out bit for bit as a reference that follows the same
// steps would produce them, so every float32 operation is rounded where it is
// written (no contraction) and the butterflies run in a fixed order: stage h
// (h = 1, 2, 4, ..., d/2) maps the pair (y_i, y_{i+h}) of each block of 2h to
// (y_i + y_{i+h}, y_i - y_{i+h}).
//
// Mapping: one CTA of 256 threads per (head, 128-row tile).  A lane holds 32
// consecutive elements of a row (d/32 lanes per row, read with 16-byte loads
// that a warp coalesces into whole rows), so stages h <= 16 run in registers
// and only h = 32 (and 64) cross lanes, by shuffle.  The tile's amax is
// reduced through shared memory, then each lane scales, converts pairs with
// cvt.rn.satfinite.e4m3x2 and writes its 32 codes with two 16-byte stores.
// Rows past N count as zeros and are not written.
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kTileRows = 128;
constexpr float kE4m3Max = 448.f;

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    // The first source goes to the upper byte.
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads)
    fp8_rotate_quantize_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                               float* __restrict__ scales, int N, int n_tiles, float inv_sqrt_d,
                               const __grid_constant__ Fp8Signs signs) {
    constexpr int L = D / 32;              // lanes per row
    constexpr int ROWS_W = 32 / L;         // rows per warp pass
    constexpr int ROWS_C = 8 * ROWS_W;     // rows per CTA pass
    constexpr int PASSES = kTileRows / ROWS_C;
    __shared__ float red[8];

    const int tile = blockIdx.x % n_tiles;
    const long long bh = blockIdx.x / n_tiles;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int part = lane % L;             // which 32 elements of the row
    const int row0 = tile * kTileRows + warp * ROWS_W + lane / L;

    float y[PASSES][32];
    // Loads first (all passes in flight), then the transform.
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int row = row0 + p * ROWS_C;
        if (row < N) {
            const uint4* src = reinterpret_cast<const uint4*>(
                x + (bh * N + row) * D + part * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 v = src[c];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    y[p][8 * c + 2 * u] = __uint_as_float(w[u] << 16);
                    y[p][8 * c + 2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) y[p][e] = 0.f;
        }
    }

    float amax = 0.f;
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
#pragma unroll
        for (int e = 0; e < 32; ++e) y[p][e] = __fmul_rn(y[p][e], signs.s[part * 32 + e]);
        // Stages h = 1 .. 16 inside the lane.
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (e & h) continue;
                const float a = y[p][e], b = y[p][e + h];
                y[p][e] = __fadd_rn(a, b);
                y[p][e + h] = __fsub_rn(a, b);
            }
        }
        // Stages h = 32 (and 64) across the lanes of the row.
#pragma unroll
        for (int m = 1; m < L; m <<= 1) {
            const bool upper = (part & m) != 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, y[p][e], m);
                y[p][e] = upper ? __fsub_rn(o, y[p][e]) : __fadd_rn(y[p][e], o);
            }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            y[p][e] = __fmul_rn(y[p][e], inv_sqrt_d);
            amax = fmaxf(amax, fabsf(y[p][e]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    const bool nz = amax > 0.f;
    const float mul = nz ? __fdiv_rn(kE4m3Max, amax) : 0.f;
    if (threadIdx.x == 0) scales[bh * n_tiles + tile] = nz ? __fdiv_rn(amax, kE4m3Max) : 1.f;

#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int row = row0 + p * ROWS_C;
        uint32_t w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint16_t lo = cvt_e4m3x2(__fmul_rn(y[p][4 * u], mul), __fmul_rn(y[p][4 * u + 1], mul));
            const uint16_t hi =
                cvt_e4m3x2(__fmul_rn(y[p][4 * u + 2], mul), __fmul_rn(y[p][4 * u + 3], mul));
            w[u] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        if (row < N) {
            uint4* dst = reinterpret_cast<uint4*>(codes + (bh * N + row) * D + part * 32);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }
}

}  // namespace

cudaError_t launch_fp8_rotate_quantize(const Fp8QuantArgs& a, cudaStream_t stream) {
    const int n_tiles = (a.N + kTileRows - 1) / kTileRows;
    const long long grid = static_cast<long long>(a.BH) * n_tiles;
    if (a.d == 64)
        fp8_rotate_quantize_kernel<64><<<static_cast<unsigned int>(grid), kQuantThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(a.x), static_cast<uint8_t*>(a.codes), a.scales, a.N,
            n_tiles, a.inv_sqrt_d, a.signs);
    else
        fp8_rotate_quantize_kernel<128><<<static_cast<unsigned int>(grid), kQuantThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(a.x), static_cast<uint8_t*>(a.codes), a.scales, a.N,
            n_tiles, a.inv_sqrt_d, a.signs);
    return cudaGetLastError();
}

}  // namespace fa
