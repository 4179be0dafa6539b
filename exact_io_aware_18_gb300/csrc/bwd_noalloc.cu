// bwd_noalloc.cu - a backward entry point that allocates no device memory.
//
// fa_bwd needs scratch space for two FP32 vectors per (batch, head): D and the
// base-2 LSE.  It takes that space from the caller or allocates it on the
// stream.  Some callers can do neither at call time: an inference or training
// runtime that reserves its whole memory budget once at start-up and may not
// allocate afterwards, or code whose device memory is owned by another
// allocator it must not bypass.  fa_bwd_noalloc serves them with scratch that
// lives in a fixed-size array inside the library itself, on every GPU that
// loads the library, for the life of the process.
//
// The array is a file-scope __device__ symbol.  Host code cannot use its name
// as a device address (on the host it is only a stand-in), so the first call
// on each device looks the address up with cudaGetSymbolAddress while that
// device is current and caches it; later calls reuse the cached pointer.
// Because of that one-time look-up, make the first call on a device before any
// stream capture begins.
//
// Every call shares the one array and leaves its contents behind.  The dQ
// step (with the first step fused) rewrites every entry that dK/dV reads
// later (padding rows included), so nothing needs clearing between calls;
// but two calls that run on the GPU at the same time (on different streams,
// say) would race on the array.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kScratchFloats = FA_NOALLOC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
float* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up once).
int scratch_ptr(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* do_, const float* lse, float* dq, float* dk, float* dv,
                              int B, int H, int N, int d, int causal, float scale, void* stream) {
    // fa_bwd's own checks first, so both entry points give the same status for
    // the same arguments; only then the size of the built-in scratch.
    if (int rc = fa::check_bwd_args(q, k, v, o, do_, lse, dq, dk, dv, B, H, N, d, scale))
        return rc;
    const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
    if (need == 0) return FA_ERR_INVALID_ARG;
    if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_NO_MEMORY;
    float* scratch = nullptr;
    if (int rc = scratch_ptr(&scratch)) return rc;
    const size_t half = need / (2 * sizeof(float));  // B*H*roundup(N,128) floats
    float* delta = scratch;
    float* lse2 = scratch + half;
    int rc = fa_bwd_dq_preprocess(q, k, v, o, do_, lse, delta, lse2, dq, B, H, N, d, causal,
                                  scale, stream);
    if (rc == FA_OK)
        rc = fa_bwd_dkdv(q, k, v, do_, delta, lse2, dk, dv, B, H, N, d, causal, scale, stream);
    return rc;
}
