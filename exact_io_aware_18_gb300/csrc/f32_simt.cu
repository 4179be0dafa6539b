// f32_simt.cu - FP32 twins of the forward and backward on CUDA cores.
//
// FP32 inputs and outputs, FP32 arithmetic with FMA, no TF32 and no tensor
// cores: these serve FP32 callers at small sizes, where the 1e-4 error bound
// of an FP32 workload rules out reduced-precision tensor-core inputs.
//
// Forward: one warp per query row; lane c holds dimensions c, c+32, ... of
// q_i and of the output accumulator.  Keys stream one at a time through the
// online-softmax update of "LLM part 06: FlashAttention - GPU SRAM, tiling
// and online softmax" (section 2) with a block of one key: m_new =
// max(m, s_j), l = l e^{m - m_new} + e^{s_j - m_new}, O likewise, and the
// division by l at the end.
//
// Backward: P is recomputed from the saved LSE ("Flash Attention:
// Revolutionizing Transformer Efficiency", section "The Flash Attention
// algorithm", recomputation).  D_i = dO_i . O_i; one warp per key row for
// dK, dV and one warp per query row for dQ, each a plain sum over the other
// side, so the FP32 backward needs no atomics and is deterministic.
#include <cmath>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 4;  // warps (rows) per block

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kWarps * 32)
    fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                   const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
                   int N, float scale) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const long long bh = blockIdx.y;
    if (i >= N) return;
    const float* qh = q + (bh * N) * D;
    const float* kh = k + (bh * N) * D;
    const float* vh = v + (bh * N) * D;
    float qi[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qi[e] = qh[static_cast<long long>(i) * D + lane + 32 * e];
        acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int last = CAUSAL ? i : N - 1;
    for (int j = 0; j <= last; ++j) {
        const float* kj = kh + static_cast<long long>(j) * D;
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) part = fmaf(qi[e], kj[lane + 32 * e], part);
        const float s = warp_sum(part) * scale;
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);  // 0 on the first key (m = -inf)
        const float p = expf(s - m_new);
        l = l * alpha + p;
        const float* vj = vh + static_cast<long long>(j) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vj[lane + 32 * e], acc[e] * alpha);
        m = m_new;
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e) o[(bh * N + i) * D + lane + 32 * e] = acc[e] * inv;
    if (lane == 0) lse[bh * N + i] = m + logf(l);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    bwd_pre_f32_kernel(const float* __restrict__ o, const float* __restrict__ dO,
                       float* __restrict__ delta, int N) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const long long bh = blockIdx.y;
    if (i >= N) return;
    const long long base = (bh * N + i) * D;
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) part = fmaf(dO[base + lane + 32 * e], o[base + lane + 32 * e], part);
    const float s = warp_sum(part);
    if (lane == 0) delta[bh * N + i] = s;
}

// dK_j = scale * sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i  (i >= j when causal)
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kWarps * 32)
    bwd_dkdv_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, const float* __restrict__ dO,
                        const float* __restrict__ lse, const float* __restrict__ delta,
                        float* __restrict__ dk, float* __restrict__ dv, int N, float scale) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const long long bh = blockIdx.y;
    if (j >= N) return;
    const long long hb = bh * N;
    float kj[E], vj[E], dkj[E], dvj[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        kj[e] = k[(hb + j) * D + lane + 32 * e];
        vj[e] = v[(hb + j) * D + lane + 32 * e];
        dkj[e] = 0.f;
        dvj[e] = 0.f;
    }
    for (int i = CAUSAL ? j : 0; i < N; ++i) {
        const float* qi = q + (hb + i) * D;
        const float* doi = dO + (hb + i) * D;
        float ps = 0.f, pd = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            ps = fmaf(qi[lane + 32 * e], kj[e], ps);
            pd = fmaf(doi[lane + 32 * e], vj[e], pd);
        }
        const float s = warp_sum(ps) * scale;
        const float dp = warp_sum(pd);
        const float p = expf(s - lse[hb + i]);
        const float ds = p * (dp - delta[hb + i]);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            dvj[e] = fmaf(p, doi[lane + 32 * e], dvj[e]);
            dkj[e] = fmaf(ds, qi[lane + 32 * e], dkj[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
        dk[(hb + j) * D + lane + 32 * e] = dkj[e] * scale;
        dv[(hb + j) * D + lane + 32 * e] = dvj[e];
    }
}

// dQ_i = scale * sum_j dS_ij k_j  (j <= i when causal)
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kWarps * 32)
    bwd_dq_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                      const float* __restrict__ v, const float* __restrict__ dO,
                      const float* __restrict__ lse, const float* __restrict__ delta,
                      float* __restrict__ dq, int N, float scale) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const long long bh = blockIdx.y;
    if (i >= N) return;
    const long long hb = bh * N;
    float qi[E], doi[E], dqi[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qi[e] = q[(hb + i) * D + lane + 32 * e];
        doi[e] = dO[(hb + i) * D + lane + 32 * e];
        dqi[e] = 0.f;
    }
    const float lse_i = lse[hb + i];
    const float d_i = delta[hb + i];
    const int last = CAUSAL ? i : N - 1;
    for (int j = 0; j <= last; ++j) {
        const float* kj = k + (hb + j) * D;
        const float* vj = v + (hb + j) * D;
        float ps = 0.f, pd = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            ps = fmaf(qi[e], kj[lane + 32 * e], ps);
            pd = fmaf(doi[e], vj[lane + 32 * e], pd);
        }
        const float s = warp_sum(ps) * scale;
        const float dp = warp_sum(pd);
        const float ds = expf(s - lse_i) * (dp - d_i);
#pragma unroll
        for (int e = 0; e < E; ++e) dqi[e] = fmaf(ds, kj[lane + 32 * e], dqi[e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) dq[(hb + i) * D + lane + 32 * e] = dqi[e] * scale;
}

template <int D, bool CAUSAL>
cudaError_t fwd_t(const F32Args& a, cudaStream_t s) {
    dim3 grid((a.N + kWarps - 1) / kWarps, a.B * a.H);
    fwd_f32_kernel<D, CAUSAL><<<grid, kWarps * 32, 0, s>>>(a.q, a.k, a.v, a.out_o, a.out_lse,
                                                           a.N, a.scale);
    return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t bwd_t(const F32Args& a, cudaStream_t s) {
    dim3 grid((a.N + kWarps - 1) / kWarps, a.B * a.H);
    bwd_pre_f32_kernel<D><<<grid, kWarps * 32, 0, s>>>(a.o, a.dO, a.delta, a.N);
    bwd_dkdv_f32_kernel<D, CAUSAL><<<grid, kWarps * 32, 0, s>>>(a.q, a.k, a.v, a.dO, a.lse,
                                                                a.delta, a.dk, a.dv, a.N,
                                                                a.scale);
    bwd_dq_f32_kernel<D, CAUSAL><<<grid, kWarps * 32, 0, s>>>(a.q, a.k, a.v, a.dO, a.lse,
                                                              a.delta, a.dq, a.N, a.scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const F32Args& a, cudaStream_t s) {
    if (a.d == 64) return a.causal ? fwd_t<64, true>(a, s) : fwd_t<64, false>(a, s);
    return a.causal ? fwd_t<128, true>(a, s) : fwd_t<128, false>(a, s);
}

cudaError_t launch_bwd_f32(const F32Args& a, cudaStream_t s) {
    if (a.d == 64) return a.causal ? bwd_t<64, true>(a, s) : bwd_t<64, false>(a, s);
    return a.causal ? bwd_t<128, true>(a, s) : bwd_t<128, false>(a, s);
}

}  // namespace fa
