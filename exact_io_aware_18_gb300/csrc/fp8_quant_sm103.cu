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
// written (no contraction; the packed two-lane instructions round each lane
// on its own) and the butterflies run in a fixed order: stage h (h = 1, 2, 4,
// ..., d/2) maps the pair (y_i, y_{i+h}) of each block of 2h to
// (y_i + y_{i+h}, y_i - y_{i+h}).
//
// Mapping: persistent CTAs of 128 threads, three per SM, each thread one row
// of the current tile, so the whole transform runs in its registers.  Two
// tile buffers per CTA: thread 0 keeps the load of the next tile in flight
// while the current one is transformed, and each tile's codes are written
// over the first half of its own buffer (its BF16 rows are all in registers
// by then) and leave by TMA store.  With 128-byte swizzled boxes on
// both sides, a warp's 16-byte shared-memory accesses to 32 different rows hit
// distinct banks.  Stages h >= 2 pair whole float2 registers and use the packed FP32
// instructions; stage 1 pairs the two halves of each float2.
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kQuantThreads = 128;  // one tile row per thread
constexpr int kQuantCtasPerSm = 3;
constexpr int kTileRows = 128;
constexpr float kE4m3Max = 448.f;

template <int D>
struct QuantCfg {
    static constexpr int KB = D / 64;             // 128-byte input boxes per bf16 row
    static constexpr int BOX_BYTES = 128 * 128;   // one 128-row x 128-byte box
    static constexpr int IN_BYTES = KB * BOX_BYTES;
    static constexpr int OUT_BYTES = 128 * D;     // one tile of codes, over its input
    static_assert(OUT_BYTES <= IN_BYTES, "the codes are written over their tile's input");
    static constexpr int NBUF = 2;
    static constexpr int OFF_IN = 0;
    static constexpr int OFF_BAR = OFF_IN + NBUF * IN_BYTES;
    static constexpr int OFF_RED = OFF_BAR + 64;
    static constexpr int LAYOUT_BYTES = OFF_RED + 64;
    static constexpr int SMEM_BYTES = LAYOUT_BYTES + 1024;  // + alignment slack
    // d = 128 codes: 128-byte rows, stored swizzled; d = 64: plain 64-byte rows.
    static constexpr bool OUT_SWIZZLED = (D == 128);
};

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    // The first source goes to the upper byte.
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads, kQuantCtasPerSm)
    fp8_rotate_quantize_kernel(const __grid_constant__ CUtensorMap tm_x,
                               const __grid_constant__ CUtensorMap tm_codes,
                               float* __restrict__ scales, int n_tiles, int n_items,
                               float inv_sqrt_d, const __grid_constant__ Fp8Signs signs,
                               unsigned int* status, unsigned long long timeout_ns) {
    using C = QuantCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    if (smem + C::LAYOUT_BYTES > smem_raw + C::SMEM_BYTES) {
        if (threadIdx.x == 0) atomicOr(status, kStatusSmemLayout);
        return;
    }
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar_full = s_base + C::OFF_BAR;  // one barrier per buffer
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBUF);
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (tid == 0) {
        for (int b = 0; b < C::NBUF; ++b) mbar_init(bar_full + 8 * b, 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_codes);
    }
    __syncthreads();
    const WaitCtx wc{status, timeout_ns, abort_flag};

    auto issue_load = [&](int item, int buf) {
        const int tile = item % n_tiles;
        const int bh = item / n_tiles;
        const uint32_t dst = s_base + C::OFF_IN + buf * C::IN_BYTES;
        mbar_arrive_expect_tx(bar_full + 8 * buf, C::IN_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(dst + kb * C::BOX_BYTES, &tm_x, bar_full + 8 * buf, kb * 64,
                        tile * kTileRows, bh);
    };
    // Tile `it` of this CTA is item blockIdx.x + it * gridDim.x, in buffer it % NBUF.
    int loads = 0;
    if (tid == 0) {
        for (int t = 0; t < C::NBUF - 1; ++t) {
            const long long item = blockIdx.x + static_cast<long long>(t) * gridDim.x;
            if (item < n_items) {
                issue_load(static_cast<int>(item), t);
                ++loads;
            }
        }
    }

    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
        const int buf = it % C::NBUF;
        if (!__syncthreads_and(mbar_wait(bar_full + 8 * buf, (it / C::NBUF) & 1, wc))) break;

        // Row `tid` of the tile: bf16 pairs -> float2 with the signs applied.
        float2 v[D / 2];
        const uint32_t in = s_base + C::OFF_IN + buf * C::IN_BYTES;
        const uint32_t out = in;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint32_t addr = in + (c >> 3) * C::BOX_BYTES + tid * 128 +
                                  ((static_cast<uint32_t>((c & 7) ^ (tid & 7))) << 4);
            uint32_t w0, w1, w2, w3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                         : "r"(addr));
            const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = 8 * c + 2 * u;
                v[e / 2] = __fmul2_rn(make_float2(__uint_as_float(w[u] << 16),
                                                  __uint_as_float(w[u] & 0xFFFF0000u)),
                                      make_float2(signs.s[e], signs.s[e + 1]));
            }
        }
        // Stage h = 1: the two halves of each float2.
#pragma unroll
        for (int i = 0; i < D / 2; i += 2) {
            const float2 a = make_float2(v[i].x, v[i + 1].x);
            const float2 b = make_float2(v[i].y, v[i + 1].y);
            const float2 s = __fadd2_rn(a, b);
            const float2 t = __ffma2_rn(b, make_float2(-1.f, -1.f), a);  // a - b, one rounding
            v[i] = make_float2(s.x, t.x);
            v[i + 1] = make_float2(s.y, t.y);
        }
        // Stages h = 2 .. D/2: float2 i pairs with float2 i + h/2.
#pragma unroll
        for (int h2 = 1; h2 < D / 2; h2 <<= 1) {
#pragma unroll
            for (int i = 0; i < D / 2; ++i) {
                if (i & h2) continue;
                const float2 a = v[i], b = v[i + h2];
                v[i] = __fadd2_rn(a, b);
                v[i + h2] = __ffma2_rn(b, make_float2(-1.f, -1.f), a);
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < D / 2; ++i) {
            v[i] = __fmul2_rn(v[i], make_float2(inv_sqrt_d, inv_sqrt_d));
            amax = fmaxf(amax, fmaxf(fabsf(v[i].x), fabsf(v[i].y)));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) red[warp] = amax;
        // Every row of this tile is in registers past this barrier: its
        // codes may overwrite it.
        __syncthreads();
        if (tid == 0) {
            // Tile it + NBUF - 1 goes to the buffer of tile it - 1, once the
            // store of tile it - 1's codes has read it.
            const long long ahead = item + static_cast<long long>(C::NBUF - 1) * gridDim.x;
            if (ahead < n_items) {
                bulk_wait_read_all();
                issue_load(static_cast<int>(ahead), (it + C::NBUF - 1) % C::NBUF);
                ++loads;
            }
        }
        amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        const bool nz = amax > 0.f;
        const float mul = nz ? __fdiv_rn(kE4m3Max, amax) : 0.f;

#pragma unroll
        for (int c = 0; c < D / 16; ++c) {  // 16 codes (one 16-byte chunk) at a time
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 p = __fmul2_rn(v[8 * c + 2 * u], make_float2(mul, mul));
                const float2 q = __fmul2_rn(v[8 * c + 2 * u + 1], make_float2(mul, mul));
                w[u] = cvt_e4m3x2(p.x, p.y) | (cvt_e4m3x2(q.x, q.y) << 16);
            }
            const uint32_t chunk = C::OUT_SWIZZLED ? (c ^ (tid & 7)) : c;
            st_shared_v4(out + tid * D + (chunk << 4), w[0], w[1], w[2], w[3]);
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            const int tile = item % n_tiles;
            const int bh = item / n_tiles;
            tma_store_3d(&tm_codes, out, 0, tile * kTileRows, bh);
            bulk_commit();
            scales[static_cast<long long>(bh) * n_tiles + tile] =
                nz ? __fdiv_rn(amax, kE4m3Max) : 1.f;
        }
    }
    if (tid == 0) {
        bulk_wait_all();
        // After an early exit prefetched tiles may still be landing.
        for (int t = it; t < loads; ++t)
            mbar_wait_drain(bar_full + 8 * (t % C::NBUF), (t / C::NBUF) & 1, timeout_ns);
    }
}

}  // namespace

cudaError_t launch_fp8_rotate_quantize(const Fp8QuantArgs& a, cudaStream_t stream) {
    const int n_tiles = (a.N + kTileRows - 1) / kTileRows;
    const long long n_items = static_cast<long long>(a.BH) * n_tiles;
    const long long cap = static_cast<long long>(kQuantCtasPerSm) * a.num_sms;
    const int grid = static_cast<int>(n_items < cap ? n_items : cap);
    if (a.d == 64) {
        auto kern = fp8_rotate_quantize_kernel<64>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             QuantCfg<64>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        kern<<<grid, kQuantThreads, QuantCfg<64>::SMEM_BYTES, stream>>>(
            *a.tm_x, *a.tm_codes, a.scales, n_tiles, static_cast<int>(n_items), a.inv_sqrt_d,
            a.signs, a.status, a.timeout_ns);
    } else {
        auto kern = fp8_rotate_quantize_kernel<128>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             QuantCfg<128>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        kern<<<grid, kQuantThreads, QuantCfg<128>::SMEM_BYTES, stream>>>(
            *a.tm_x, *a.tm_codes, a.scales, n_tiles, static_cast<int>(n_items), a.inv_sqrt_d,
            a.signs, a.status, a.timeout_ns);
    }
    return cudaGetLastError();
}

}  // namespace fa
