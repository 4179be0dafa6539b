// fa_internal.h - launch descriptors shared between the C-ABI layer
// (fa_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace fa {

// Launches kern with programmatic stream serialization: its CTAs may be
// scheduled while the kernel before it in the stream finishes (on the SMs
// that kernel's CTAs leave).  The kernel itself waits for its predecessor
// (pdl_wait_then_release, sm103_primitives.cuh) before it touches global
// memory, so only its launch and set-up overlap.
template <typename... Params, typename... Args>
cudaError_t launch_overlapped(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Heads per claim group of the persistent kernels.  Their work items are
// claimed a group of heads at a time, heaviest first inside the group, so
// that the group's shared operands stay in L2: about 128 tiles per group, 256
// under a causal mask from 32 tiles per head on (measured faster there, and
// slower at 16 tiles or without the mask).
inline int claim_group(int n_tiles, bool causal) {
    const int g = ((causal && n_tiles >= 32) ? 256 : 128) / n_tiles;
    return g < 1 ? 1 : g;
}

// Forward (BF16).  Tensor maps view Q, K, V, O as 3-D arrays
// (d, N, B*H) of bf16 with 128 x 64 boxes and 128-byte swizzle.
struct FwdArgs {
    const CUtensorMap* tm_q;
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    const CUtensorMap* tm_o;
    float* lse;
    int B, H, N, d;    // H query heads
    int Hkv;           // K/V heads, H = n_rep * Hkv (grouped-query attention)
    int causal;
    float scale_log2;  // scale * log2(e)
    unsigned int* status;
    unsigned long long timeout_ns;
    unsigned int* work;  // tile counter of this launch, zero between launches
    int num_sms;         // persistent grid size
    // Split-KV (decode): N is the number of queries, Nk the number of keys;
    // key tiles are cut into n_splits chunks of chunk_tiles, and each (head,
    // Q tile, chunk) writes its normalised FP32 partial O and natural-log LSE
    // to o_part [n_splits][B*H][N][d] and lse_part [n_splits][B*H][N].  The
    // plain forward has Nk = N, n_splits = 1 and no partial buffers.
    int Nk;
    int n_splits;
    int chunk_tiles;
    float* o_part;
    float* lse_part;
    // FP8 forward: tm_q and tm_k view E4M3 codes (d, N, B*H) with one 128 x d
    // box; q_scale [B*H][ceil(N/128)] and k_scale [B*Hkv][ceil(N/128)] are the
    // tiles' dequantisation scales.  Null for the BF16 forward.
    const float* q_scale;
    const float* k_scale;
};

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_splitkv_bf16(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream);

// Rotation by diag(s) H / sqrt(d) and per-128-row-tile E4M3 quantisation of
// one BF16 tensor [BH][N][d]: codes [BH][N][d] (bytes), scales [BH][ceil(N/128)].
// tm_x views x like the forward's BF16 maps; tm_codes views the codes as
// (d, N, BH) bytes with one 128-row box (128-byte swizzle at d = 128, none at
// d = 64).
struct Fp8Signs {
    float s[128];  // +1 / -1, the first d entries used
};

struct Fp8QuantArgs {
    const CUtensorMap* tm_x;
    const CUtensorMap* tm_codes;
    float* scales;
    int BH, N, d;
    float inv_sqrt_d;  // float32 value of 1 / sqrt(d)
    Fp8Signs signs;
    unsigned int* status;
    unsigned long long timeout_ns;
    int num_sms;
};

cudaError_t launch_fp8_rotate_quantize(const Fp8QuantArgs& a, cudaStream_t stream);

// Merge of the split-KV partials: per query row, O = sum_s w_s O_s / sum_s w_s
// and LSE = m + ln sum_s w_s with w_s = exp(LSE_s - m), m = max_s LSE_s;
// O is written as BF16 [BH][N][d], LSE as FP32 [BH][N].
struct CombineArgs {
    const float* o_part;
    const float* lse_part;
    void* o;
    float* lse;
    int BH, N, d, n_splits;
};

cudaError_t launch_splitkv_combine(const CombineArgs& a, cudaStream_t stream);

// Backward preprocess (BF16): D and base-2 LSE into padded [B*H, n_pad]
// vectors.
struct BwdPreArgs {
    const void* o;
    const void* dO;
    const float* lse;
    float* delta;
    float* lse2;
    int BH, N, d, n_pad;
};

cudaError_t launch_bwd_pre_bf16(const BwdPreArgs& a, cudaStream_t stream);

// Backward dK/dV (BF16).  Tensor maps for Q, K, V, dO as for the forward;
// dK and dV through FP32 maps (d, N, B*H) with 32 x 32 boxes, 128-byte swizzle.
struct BwdArgs {
    const CUtensorMap* tm_q;
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    const CUtensorMap* tm_do;
    const CUtensorMap* tm_dk;
    const CUtensorMap* tm_dv;
    const float* delta;
    const float* lse2;
    int B, H, N, d, n_pad;  // H query heads
    int Hkv;                // K/V heads, H = n_rep * Hkv
    int causal;
    float scale;       // multiplies dS (dQ = dS K, dK = dS^T Q with dS scaled)
    float scale_log2;  // scale * log2(e), for recomputing P
    unsigned int* status;
    unsigned long long timeout_ns;
    unsigned int* work;  // tile counter of this launch, zero between launches
    int num_sms;         // persistent grid size
};

cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t stream);

// Backward dQ (BF16): persistent CTAs that claim Q tiles, a loop over key
// tiles per Q tile, dq written once (FP32, from a staging box per warp).
struct DqArgs {
    const CUtensorMap* tm_q;
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    const CUtensorMap* tm_do;
    float* dq;  // FP32 [B,H,N,d], 16-byte aligned
    // o (bf16 [B,H,N,d]) and lse (float [B,H,N]) non-null: the kernel also
    // does the first backward step and writes delta and lse2; null: it reads
    // them as that step wrote them.  tm_o views o like tm_q views q (null
    // when o is).
    const void* o;
    const CUtensorMap* tm_o;
    const float* lse;
    float* delta;
    float* lse2;
    int B, H, N, d, n_pad;  // H query heads
    int Hkv;                // K/V heads, H = n_rep * Hkv
    int causal;
    float scale;
    float scale_log2;
    unsigned int* status;
    unsigned long long timeout_ns;
    unsigned int* work;  // tile counter of this launch, zero between launches
    int num_sms;         // persistent grid size
};

cudaError_t launch_bwd_dq_bf16(const DqArgs& a, cudaStream_t stream);

// FP32 SIMT twins.
struct F32Args {
    const float* q;
    const float* k;
    const float* v;
    const float* o;
    const float* dO;
    const float* lse;
    float* out_o;
    float* out_lse;
    float* dq;
    float* dk;
    float* dv;
    float* delta;
    int B, H, N, d;
    int causal;
    float scale;
};

cudaError_t launch_fwd_f32(const F32Args& a, cudaStream_t stream);
cudaError_t launch_bwd_f32(const F32Args& a, cudaStream_t stream);

// The argument checks fa_bwd makes before it looks at its workspace (null
// and misaligned pointers, sizes, head dimension, scale), in the same order
// and with the same status codes; fa_bwd_noalloc runs them first too.
int check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* do_,
                   const float* lse, const float* dq, const float* dk, const float* dv, int B,
                   int H, int N, int d, float scale);

// Failure-detection self-test kernel (waits on a barrier nobody arrives at).
cudaError_t launch_wait_timeout_selftest(unsigned int* status, unsigned long long timeout_ns,
                                         cudaStream_t stream);

}  // namespace fa
