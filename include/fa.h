/*
 * fa.h - C ABI of the GB300 (sm_103a) exact-attention library libfa.so.
 *
 * Operation.  For every batch b and head h, with S = scale * Q K^T:
 *
 *     O   = softmax(S [+ causal mask]) V
 *     LSE = per-row natural-log logsumexp of the (masked) row of S
 *
 * (standard attention as restated in "Flash Attention: Revolutionizing
 * Transformer Efficiency", section "Standard attention: a quick recap"), and
 * its gradient dQ, dK, dV.  The forward is computed tile by tile with the
 * online-softmax running max and running sum ("LLM part 06: FlashAttention -
 * GPU SRAM, tiling and online softmax", section 2), so the N x N score matrix
 * never reaches device memory; the backward recomputes the probabilities from
 * the saved LSE ("Flash Attention: Revolutionizing Transformer Efficiency",
 * section "The Flash Attention algorithm", idea 2, recomputation).
 *
 * Conventions shared by every entry point:
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are [B, H, N, d] row-major and
 *     contiguous; LSE is [B, H, N].  Queries and keys have the same length N.
 *   - Causal (causal != 0): key j is visible to query i iff j <= i.
 *   - scale multiplies Q K^T before the softmax; it must be finite and > 0
 *     (the usual value is 1/sqrt(d)).
 *   - All pointers are DEVICE pointers into memory of the current CUDA
 *     device, owned by the caller; the library never frees them.  Every
 *     pointer must be 16-byte aligned.
 *   - stream is a cudaStream_t passed as void* (NULL: the legacy default
 *     stream).  Work is enqueued on it and the call returns without waiting.
 *     The tensor-core forward and backward kernels are launched with
 *     programmatic stream serialization: their CTAs may be scheduled and set
 *     up while the kernel before them in the stream finishes, but each waits
 *     for that kernel to complete before it reads or writes any global
 *     memory, so the stream's ordering is the same as for plain launches
 *     (also inside a captured CUDA graph).
 *   - Return value: FA_OK, or a negative fa_status.  Argument errors
 *     (INVALID_ARG, UNSUPPORTED, MISALIGNED) are found before anything is
 *     launched.  FA_ERR_CUDA reports a launch error.  A kernel that gives up
 *     on a bounded wait records FA_ERR_DEVICE_TIMEOUT in the library's device
 *     status word, read with fa_device_status().
 *   - The library holds no state between calls other than the per-device
 *     status word, a cached driver entry point and the scratch array of
 *     fa_bwd_noalloc; calls are thread-safe as long as their buffers do not
 *     overlap (fa_bwd_noalloc calls share one array, see there).
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1,    /* null pointer, non-positive size, bad scale  */
    FA_ERR_UNSUPPORTED = -2,    /* head dimension or size outside what is built */
    FA_ERR_MISALIGNED = -3,     /* a pointer is not 16-byte aligned            */
    FA_ERR_CUDA = -4,           /* a CUDA runtime/driver call or launch failed */
    FA_ERR_DEVICE_TIMEOUT = -5, /* a kernel gave up on a bounded wait          */
    FA_ERR_NO_MEMORY = -6,      /* workspace too small or allocation failed    */
} fa_status;

/* Forward, BF16 inputs and output, FP32 accumulation.
 *
 * q, k, v : const bf16 [B,H,N,d];  o : bf16 [B,H,N,d] (written);
 * lse     : float [B,H,N] (written), natural log.
 * d must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise).  N may be any value
 * >= 1: the ragged last tile is masked.  B, H <= 65535.
 *
 * One persistent CTA per SM takes 128-row Q tiles of (b, h) in turn and
 * streams the 128-key K/V tiles through a shared-memory ring ("FlashAttention
 * scaling, multi-GPU training and weight quantization", section 1: loop order
 * with Q outside, parallelism over the sequence, asynchronous TMA copies);
 * the 1/l normalisation is applied once at the end ("FlashAttention-2",
 * technical architecture, improvement 1). */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, int causal, float scale, void* stream);

/* Bytes of device workspace fa_bwd needs: two FP32 vectors per (b, h) of
 * length N rounded up to 128 (D = rowsum(dO o O) and LSE in base 2). */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/* Backward, BF16 inputs, FP32 gradients.
 *
 * q, k, v, o, do_ : const bf16 [B,H,N,d]  (o and lse as written by fa_fwd);
 * lse             : const float [B,H,N];
 * dq, dk, dv      : float [B,H,N,d] (written).
 * workspace       : device buffer of at least fa_bwd_workspace_bytes() bytes,
 *                   16-byte aligned, or NULL: the library then allocates and
 *                   frees it on the stream (cudaMallocAsync / cudaFreeAsync).
 *
 * Runs fa_bwd_dq_preprocess, then fa_bwd_dkdv, on the stream.  Every
 * gradient entry is one sum in a fixed order (no atomics), so repeated calls
 * give identical bits. */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* do_,
           const float* lse, float* dq, float* dk, float* dv,
           int B, int H, int N, int d, int causal, float scale,
           void* workspace, size_t workspace_bytes, void* stream);

/* First backward step.  delta_ws : float [B*H, roundup(N,128)] receives
 * D_i = sum_c dO_ic O_ic (0 on padding rows); lse2_ws (same shape) receives
 * LSE_i * log2(e) (+inf on padding rows).  Memory-bound; d must be 64 or 128. */
int fa_bwd_preprocess(const void* o, const void* do_, const float* lse, float* delta_ws,
                      float* lse2_ws, int B, int H, int N, int d, void* stream);

/* Second backward step, dK and dV.  One CTA per 128-key K/V tile of one
 * (b, h): it keeps K, V and the dK, dV accumulators on chip and loops over
 * the Q tiles that see those keys, recomputing P from lse2_ws ("Flash
 * Attention: Revolutionizing Transformer Efficiency", section "The Flash
 * Attention algorithm", recomputation; "FlashAttention-2", technical
 * architecture, improvement 2, parallelism over the sequence).
 * delta_ws / lse2_ws as written by fa_bwd_preprocess or fa_bwd_dq_preprocess;
 * dk, dv float [B,H,N,d]. */
int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* do_,
                const float* delta_ws, const float* lse2_ws, float* dk, float* dv,
                int B, int H, int N, int d, int causal, float scale, void* stream);

/* Third backward step, dQ.  One CTA per 128-row Q tile of one (b, h): it
 * loops over the key tiles that Q tile sees (the forward's loop order),
 * recomputes P and dP and accumulates dQ on chip, then writes each dq row
 * once (float [B,H,N,d]).  Inputs as for fa_bwd_dkdv. */
int fa_bwd_dq(const void* q, const void* k, const void* v, const void* do_,
              const float* delta_ws, const float* lse2_ws, float* dq,
              int B, int H, int N, int d, int causal, float scale, void* stream);

/* fa_bwd_dq with the first step fused into it: each dQ CTA, which already
 * holds its dO tile in shared memory, also reads its 128 rows of O and LSE,
 * forms D_i = sum_c dO_ic O_ic and LSE_i log2(e), uses them, and writes them
 * to delta_ws / lse2_ws exactly as fa_bwd_preprocess would (padding rows
 * included), ready for fa_bwd_dkdv.  The backward is then two launches: this
 * call, then fa_bwd_dkdv.  o, lse as for fa_bwd (non-null, else
 * FA_ERR_INVALID_ARG); other arguments as for fa_bwd_dq.  D's summation order
 * differs from fa_bwd_preprocess's, so the two agree to FP32 rounding, not
 * bit for bit; each is deterministic. */
int fa_bwd_dq_preprocess(const void* q, const void* k, const void* v, const void* o,
                         const void* do_, const float* lse, float* delta_ws, float* lse2_ws,
                         float* dq, int B, int H, int N, int d, int causal, float scale,
                         void* stream);

/* Grouped-query attention ("FlashAttention-2", variants: multi-query and
 * grouped-query attention): Hq query heads share Hkv K/V heads, Hq = g * Hkv,
 * and query head h attends with K/V head h / g (Hkv = 1 is multi-query
 * attention; Hkv = Hq is fa_fwd / fa_bwd).  Hkv must divide Hq, else
 * FA_ERR_INVALID_ARG.
 *
 * q, o, do_, dq : [B,Hq,N,d];  k, v, dk, dv : [B,Hkv,N,d];  lse : [B,Hq,N].
 * Types, workspace (fa_bwd_workspace_bytes(B, Hq, N, d)), errors and
 * determinism as for fa_fwd / fa_bwd.  The K/V tile loads of the forward
 * and the dQ step read the group's head; the dK/dV step runs one CTA per key
 * tile of each K/V head and sums over the Q tiles of all g query heads, so
 * dk and dv are still written once. */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* do_,
               const float* lse, float* dq, float* dk, float* dv,
               int B, int Hq, int Hkv, int N, int d, int causal, float scale,
               void* workspace, size_t workspace_bytes, void* stream);

/* Split-KV forward for decode-like shapes: few queries per head (Nq), many
 * keys (Nk).  Every query attends to all Nk keys (no mask: the new tokens
 * read the whole cache).  The key tiles are cut into n_splits chunks; each
 * (head, 128-query tile, chunk) is computed like the forward and leaves its
 * normalised FP32 partial output and LSE in the workspace, then a merge
 * kernel combines the chunks with the block merge of "LLM part 06:
 * FlashAttention - GPU SRAM, tiling and online softmax", section 2:
 * O = sum_s w_s O_s / sum_s w_s, LSE = m + ln sum_s w_s, w_s = exp(LSE_s - m),
 * m = max_s LSE_s.  The result equals fa_fwd_gqa with Nq queries and Nk keys,
 * non-causal, up to rounding.
 *
 * q, o : bf16 [B,Hq,Nq,d];  k, v : bf16 [B,Hkv,Nk,d];  lse : float [B,Hq,Nq].
 * Hkv divides Hq (grouped-query attention; Hkv = Hq for multi-head).
 * The g = Hq / Hkv query heads of a K/V head share its tiles: their g * Nq
 * query rows (contiguous in q) are computed together, 128 rows at a time,
 * so each K/V tile is read once per group.
 * n_splits <= 0 lets the library choose: the count that minimises waves x
 * (key tiles per chunk + 2) for the (K/V head, 128-query tile, chunk) items
 * over the SMs, so that the items fill whole waves; the count actually used
 * never leaves a chunk empty and is at most the number of 128-key tiles.
 * workspace : device buffer of at least
 *             fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, n_splits)
 *             bytes, 16-byte aligned, or NULL: the library then allocates and
 *             frees it on the stream.  Returns 0 for invalid sizes. */
size_t fa_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                      int n_splits);
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int n_splits,
                   void* workspace, size_t workspace_bytes, void* stream);

/* FP8 forward ("FlashAttention scaling, multi-GPU training and weight
 * quantization", section 1, FlashAttention-3, FP8 low-precision support):
 * block quantisation, each small tile with its own scale, and incoherent
 * processing, Q and K multiplied by a random orthogonal matrix before they are
 * quantised.  Two calls: fa_fp8_quantize once for Q and once for K, then
 * fa_fwd_fp8.
 *
 * fa_fp8_quantize: y = x R with R = diag(signs) H / sqrt(d) (H the Sylvester
 * Hadamard matrix, so R is orthogonal and Q R (K R)^T = Q K^T), then per
 * 128-row tile of each head, with amax = max |y| over the tile:
 *     codes = E4M3(y * (448 / amax)), round to nearest even, saturating;
 *     scale = amax / 448  (an all-zero tile: codes 0, scale 1).
 * All float32 steps are rounded in that order (the butterflies of the
 * transform in stages h = 1, 2, 4, ...: (y_i, y_i+h) -> (y_i + y_i+h,
 * y_i - y_i+h)), so the codes are reproducible bit for bit.
 *   x      : device, bf16 [BH, N, d], 16-byte aligned; d = 64 or 128.
 *   signs  : HOST array of d floats, each +1 or -1 (FA_ERR_INVALID_ARG
 *            otherwise); read during the call only.
 *   codes  : device, E4M3 bytes [BH, N, d], 16-byte aligned.
 *   scales : device, float [BH, ceil(N / 128)], 16-byte aligned.
 *
 * fa_fwd_fp8: attention with S = (Q R)(K R)^T computed from the codes on the
 * FP8 tensor cores (FP32 accumulation) and multiplied by the Q and K tile
 * scales; P V in BF16 as in fa_fwd.  Output O (bf16 [B,Hq,N,d]) and LSE
 * (float [B,Hq,N]) as fa_fwd_gqa.  d is 64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 *   q8, q_scale : fa_fp8_quantize of q [B,Hq,N,d] (BH = B*Hq).
 *   k8, k_scale : fa_fp8_quantize of k [B,Hkv,N,d] with the same signs.
 *   v           : bf16 [B,Hkv,N,d], not rotated.
 * All device pointers 16-byte aligned. */
int fa_fp8_quantize(const void* x, const float* signs, void* codes, float* scales,
                    int BH, int N, int d, void* stream);
int fa_fwd_fp8(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
               const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
               int causal, float scale, void* stream);

/* Size of the scratch array built into the library for fa_bwd_noalloc:
 * 8 MiB, i.e. B * H * roundup(N, 128) <= 1048576. */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* Backward that allocates no device memory (the pages have no counterpart:
 * this is a service to callers, not a step of the method).  For callers that
 * cannot allocate at call time: runtimes that reserve their whole device
 * memory budget at start-up, or code whose memory belongs to an allocator it
 * must not bypass.  Same arguments and results as fa_bwd, minus the
 * workspace: the D / LSE2 scratch lives in an array of
 * FA_NOALLOC_SCRATCH_BYTES inside the library, held on every GPU that loads
 * the library until the process exits.  Returns FA_ERR_NO_MEMORY, before
 * launching anything, when 2 * 4 * B * H * roundup(N,128) bytes exceed it.
 * The first call on a device looks the array's device address up
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the array and it keeps the last
 * call's contents (every entry a call reads is first written by that call);
 * calls that overlap on the GPU race on it. */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* do_,
                   const float* lse, float* dq, float* dk, float* dv,
                   int B, int H, int N, int d, int causal, float scale, void* stream);

/* FP32 twins (FP32 inputs and outputs, FP32 arithmetic on CUDA cores, no
 * TF32).  Same shapes and conventions as the BF16 calls; d is 64 or 128.
 * fa_bwd_f32's workspace holds D: at least fa_bwd_workspace_bytes() bytes,
 * or NULL to let the library allocate it on the stream. */
int fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
               int B, int H, int N, int d, int causal, float scale, void* stream);
int fa_bwd_f32(const float* q, const float* k, const float* v, const float* o,
               const float* do_, const float* lse, float* dq, float* dk, float* dv,
               int B, int H, int N, int d, int causal, float scale,
               void* workspace, size_t workspace_bytes, void* stream);

/* Static description of an fa_status value (never NULL). */
const char* fa_error_string(int status);

/* Synchronises the current device, then returns FA_ERR_DEVICE_TIMEOUT if a
 * kernel of this library has recorded a bounded-wait timeout on it since the
 * last clear, FA_ERR_CUDA if the synchronisation itself failed, else FA_OK.
 * clear != 0 resets the word. */
int fa_device_status(int clear);

/* The same check without clearing the word: fa_device_status(0). */
int fa_last_device_status(void);

/* Upper bound, in nanoseconds, on any single wait inside a kernel launched
 * after this call (default 4e9).  Values below 1e6 are raised to 1e6. */
void fa_set_wait_timeout_ns(unsigned long long ns);

/* Failure-detection self-test: launches one CTA that waits on a barrier no
 * thread ever arrives at, bounded by timeout_ns, and synchronises.  Returns
 * FA_ERR_DEVICE_TIMEOUT when the kernel gave up and reported it (the
 * expected outcome), FA_OK if the wait somehow completed, FA_ERR_CUDA on a
 * CUDA error.  Does not touch the status word read by fa_device_status. */
int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
