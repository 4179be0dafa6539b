// splitkv_combine_sm103.cu - merge of the split-KV partial results of the
// decode forward (memory-bound).
//
// Key chunk s of a query row left O_s, the softmax-weighted mean of its keys'
// values (normalised within the chunk), and LSE_s, the natural log of its sum
// of exponentials.  The result over all keys follows from the block merge of
// "LLM part 06: FlashAttention - GPU SRAM, tiling and online softmax"
// (section 2), written for normalised blocks: with m = max_s LSE_s and
// w_s = exp(LSE_s - m),
//     O   = sum_s w_s O_s / sum_s w_s,      LSE = m + ln sum_s w_s.
// One warp per query row: lanes take the split LSEs in strides and reduce the
// max by shuffles, then each lane merges d/32 consecutive elements of O (16-
// or 8-byte loads, so a warp reads each partial row in one 512- or 256-byte
// transaction) and writes them as BF16.  The partials are read eight chunks
// at a time, all loads first: one at a time, each chunk would wait for its own
// L2 round trip.
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kSplitBatch = 8;  // chunks whose partials are loaded together

template <int D>
__global__ void __launch_bounds__(kCombineThreads)
    splitkv_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                           __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                           long long rows, int n_splits) {
    constexpr int E = D / 32;  // elements of a row per lane
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (kCombineThreads / 32);
    for (long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
         row < rows; row += warps) {
        float m = -INFINITY;
        for (int s = lane; s < n_splits; s += 32) m = fmaxf(m, lse_part[s * rows + row]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        float wsum = 0.f;
        for (int s0 = 0; s0 < n_splits; s0 += kSplitBatch) {
            float lw[kSplitBatch];
            float x[kSplitBatch][E];
#pragma unroll
            for (int u = 0; u < kSplitBatch; ++u) {
                const int s = s0 + u;
#pragma unroll
                for (int e = 0; e < E; ++e) x[u][e] = 0.f;
                lw[u] = -INFINITY;  // a missing chunk weighs exp(-inf) = 0
                if (s < n_splits) {
                    lw[u] = lse_part[s * rows + row];
                    const float* src = o_part + (s * rows + row) * D + lane * E;
                    if constexpr (E == 4) {
                        const float4 v = *reinterpret_cast<const float4*>(src);
                        x[u][0] = v.x;
                        x[u][1] = v.y;
                        x[u][2] = v.z;
                        x[u][3] = v.w;
                    } else {
                        const float2 v = *reinterpret_cast<const float2*>(src);
                        x[u][0] = v.x;
                        x[u][1] = v.y;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kSplitBatch; ++u) {
                if (s0 + u >= n_splits) break;
                const float w = expf(lw[u] - m);
                wsum += w;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(w, x[u][e], acc[e]);
            }
        }
        const float inv = 1.f / wsum;
        __nv_bfloat16* dst = o + row * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<__nv_bfloat162*>(dst + e) =
                __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
        if (lane == 0) lse[row] = m + logf(wsum);
    }
}

}  // namespace

cudaError_t launch_splitkv_combine(const CombineArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.BH) * a.N;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long want = (rows + kCombineThreads / 32 - 1) / (kCombineThreads / 32);
    const long long cap = static_cast<long long>(sms) * 8;
    const int grid = static_cast<int>(want < cap ? want : cap);
    auto* o = static_cast<__nv_bfloat16*>(a.o);
    if (a.d == 64)
        splitkv_combine_kernel<64><<<grid, kCombineThreads, 0, stream>>>(
            a.o_part, a.lse_part, o, a.lse, rows, a.n_splits);
    else
        splitkv_combine_kernel<128><<<grid, kCombineThreads, 0, stream>>>(
            a.o_part, a.lse_part, o, a.lse, rows, a.n_splits);
    return cudaGetLastError();
}

}  // namespace fa
