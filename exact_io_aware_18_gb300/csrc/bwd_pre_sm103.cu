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
// a row and reduce with warp shuffles.  A warp owns 32 / (d/8) consecutive
// rows per group and issues the loads of two groups (LSE included) before it
// reduces any, so that enough bytes are in flight to keep HBM busy and no
// load waits on another; warps stride over the rows with the whole grid (at
// most full occupancy on every SM).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kPreThreads = 256;
constexpr int kPreGroups = 2;

template <int D>
__global__ void __launch_bounds__(kPreThreads)
    bwd_pre_bf16_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                        const float* __restrict__ lse, float* __restrict__ delta,
                        float* __restrict__ lse2, int N, int n_pad,
                        long long total_rows) {
    constexpr int TPR = D / 8;          // threads per row
    constexpr int RW = 32 / TPR;        // rows per warp and group
    constexpr int U = kPreGroups;       // groups whose loads are in flight together
    const int lane = threadIdx.x & 31;
    const int sub = lane % TPR;
    const long long warp_id = (static_cast<long long>(blockIdx.x) * kPreThreads + threadIdx.x) / 32;
    const long long n_warps = static_cast<long long>(gridDim.x) * (kPreThreads / 32);
    // total_rows is a multiple of 128 and RW * U divides 128, so every row of
    // a warp's batch exists and the shuffles below see the whole warp.
    for (long long r0 = warp_id * (RW * U); r0 < total_rows; r0 += n_warps * (RW * U)) {
        uint4 a[U], b[U];
        float l[U];
        bool real[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long r = r0 + u * RW + lane / TPR;
            // n_pad is a multiple of 128 and r / 128 fits 32 bits (tiles x
            // heads < 2^31): a 32-bit division finds the head.
            const unsigned int tr = static_cast<unsigned int>(r >> 7);
            const unsigned int bh = tr / static_cast<unsigned int>(n_pad >> 7);
            const int i = static_cast<int>(r - static_cast<long long>(bh) * n_pad);
            real[u] = i < N;
            const long long row = static_cast<long long>(bh) * N + i;
            if (real[u]) {
                a[u] = o[row * (D / 8) + sub];
                b[u] = dO[row * (D / 8) + sub];
                l[u] = lse[row];
            } else {
                a[u] = make_uint4(0u, 0u, 0u, 0u);
                b[u] = a[u];
                l[u] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[u]);
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = __bfloat1622float2(a2[e]);
                const float2 y = __bfloat1622float2(b2[e]);
                part = fmaf(x.x, y.x, part);
                part = fmaf(x.y, y.y, part);
            }
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1)
                part += __shfl_xor_sync(0xffffffffu, part, off);
            if (sub == 0) {
                const long long r = r0 + u * RW + lane / TPR;
                delta[r] = real[u] ? part : 0.f;
                lse2[r] = real[u] ? l[u] * 1.4426950408889634f : INFINITY;
            }
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
    const int rows_per_block = (kPreThreads / 32) * (32 / (a.d / 8)) * kPreGroups;
    long long blocks = (total + rows_per_block - 1) / rows_per_block;
    auto kern = a.d == 64 ? bwd_pre_bf16_kernel<64> : bwd_pre_bf16_kernel<128>;
    // One wave: as many blocks as are resident at once, striding over the rows.
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPreThreads, 0) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    const long long cap = static_cast<long long>(sms) * per_sm;
    if (blocks > cap) blocks = cap;
    kern<<<static_cast<int>(blocks), kPreThreads, 0, stream>>>(
        static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dO), a.lse, a.delta, a.lse2,
        a.N, a.n_pad, total);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(unsigned int* status, unsigned long long timeout_ns,
                                         cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace fa
