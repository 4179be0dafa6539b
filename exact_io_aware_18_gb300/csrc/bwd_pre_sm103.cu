// bwd_pre_sm103.cu - first step of the attention backward (memory-bound), and
// the failure-detection self-test kernel.
//
// For every (b, h) and query row i (padded up to a multiple of 128):
//   delta[i] = D_i = sum_c dO_ic O_ic     (0 on padding rows)
//   lse2[i]  = LSE_i * log2(e)            (+inf on padding rows, so that the
//                                          recomputed P of a padding row is 0)
// D is the row term of the softmax gradient dS = P o (dP - D); P itself is
// recomputed later from LSE ("Flash Attention: Revolutionizing Transformer
// Efficiency", section "The Flash Attention algorithm", recomputation).
//
// Each thread reads 16-byte vectors, 8 bf16 of O and of dO; d/8 threads share
// a row and reduce with warp shuffles.  The grid is
// a multiple of the SM count with a grid-stride loop over rows.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kPreThreads = 256;

template <int D>
__global__ void __launch_bounds__(kPreThreads)
    bwd_pre_bf16_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                        const float* __restrict__ lse, float* __restrict__ delta,
                        float* __restrict__ lse2, int N, int n_pad,
                        long long total_rows) {
    constexpr int TPR = D / 8;                  // threads per row
    constexpr int RPB = kPreThreads / TPR;      // rows per block per pass
    const int sub = threadIdx.x % TPR;
    for (long long r = static_cast<long long>(blockIdx.x) * RPB + threadIdx.x / TPR;
         r < total_rows; r += static_cast<long long>(gridDim.x) * RPB) {
        const long long bh = r / n_pad;
        const int i = static_cast<int>(r - bh * n_pad);
        float part = 0.f;
        const bool real = i < N;
        if (real) {
            const long long row = bh * N + i;
            const uint4 a = o[row * (D / 8) + sub];
            const uint4 b = dO[row * (D / 8) + sub];
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = __bfloat1622float2(a2[e]);
                const float2 y = __bfloat1622float2(b2[e]);
                part = fmaf(x.x, y.x, part);
                part = fmaf(x.y, y.y, part);
            }
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1)
            part += __shfl_xor_sync(0xffffffffu, part, off);
        if (sub == 0) {
            delta[r] = real ? part : 0.f;
            lse2[r] = real ? lse[bh * N + i] * 1.4426950408889634f : INFINITY;
        }
    }
}

__global__ void wait_timeout_selftest_kernel(unsigned int* status,
                                             unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    const uint32_t bar = smem_u32(&bar_storage);
    mbar_init(bar, 1);
    abort_flag = 0;
    mbar_fence_init();
    // Nobody arrives: the bounded wait must give up and report it.
    const WaitCtx wc{status, timeout_ns, &abort_flag};
    mbar_wait(bar, 0, wc);
}

}  // namespace

cudaError_t launch_bwd_pre_bf16(const BwdPreArgs& a, cudaStream_t stream) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = static_cast<long long>(a.BH) * a.n_pad;
    const int rpb = kPreThreads / (a.d / 8);
    long long blocks = (total + rpb - 1) / rpb;
    const long long cap = static_cast<long long>(sms) * 16;
    if (blocks > cap) blocks = cap;
    if (a.d == 64)
        bwd_pre_bf16_kernel<64><<<static_cast<int>(blocks), kPreThreads, 0, stream>>>(
            static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dO), a.lse, a.delta,
            a.lse2, a.N, a.n_pad, total);
    else
        bwd_pre_bf16_kernel<128><<<static_cast<int>(blocks), kPreThreads, 0, stream>>>(
            static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dO), a.lse, a.delta,
            a.lse2, a.N, a.n_pad, total);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(unsigned int* status, unsigned long long timeout_ns,
                                         cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace fa
