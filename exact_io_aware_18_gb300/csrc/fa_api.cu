// fa_api.cu - the C ABI of libfa.so (declared in include/fa.h): argument
// checks, TMA tensor-map encoding, workspace handling and kernel dispatch.
// Nothing here computes attention; every numeric step runs in the kernels.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// Device status word: kernels OR kStatusTimeout into it when a bounded wait
// gives up.  One copy per device (a __device__ variable is per context).
__device__ unsigned int g_fa_status;

std::atomic<unsigned long long> g_timeout_ns{4000000000ull};

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};
std::mutex g_mutex;

// Tile counters of the persistent kernels.  Each launch takes the next slot
// of a ring (two words, the second spare); the CTA that makes the launch's
// last claim puts the counter back to zero, so launches that overlap on
// different streams use different slots (up to kWorkSlots in flight).
constexpr int kWorkSlots = 256;
__device__ unsigned int g_fa_work[2 * kWorkSlots];
unsigned int* g_work_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::atomic<unsigned int> g_work_next{0};

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;

int status_ptr(unsigned int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    *out = g_status_ptr[dev];
    return FA_OK;
}

// A tile-counter pair for one launch and the SM count of the current device.
int work_slot(unsigned int** out, int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!g_work_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_fa_work) != cudaSuccess) return FA_ERR_CUDA;
            int n = 0;
            if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                n < 1)
                return FA_ERR_CUDA;
            g_work_ptr[dev] = static_cast<unsigned int*>(p);
            g_num_sms[dev] = n;
        }
    }
    const unsigned int slot = g_work_next.fetch_add(1) % kWorkSlots;
    *out = g_work_ptr[dev] + 2 * slot;
    *sms = g_num_sms[dev];
    return FA_OK;
}

int get_encode(EncodeFn* out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return FA_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeFn>(fn);
    }
    *out = g_encode;
    return FA_OK;
}

// [B*H, N, d] bf16 viewed as (d, N, B*H); 128-row x 64-column boxes (128 bytes
// wide, the 128-byte swizzle span).  Rows past N read as zero, stores past N
// are dropped.
int make_map_bf16(CUtensorMap* map, const void* ptr, int d, int N, long long BH) {
    EncodeFn enc;
    if (int rc = get_encode(&enc)) return rc;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// [B*H, N, d] E4M3 codes (bytes) viewed as (d, N, B*H) with one 128-row box
// of d bytes: 128-byte swizzle at d = 128 (exactly its span); at d = 64 none
// (the quantisation kernel's plain stores) or, for MMA operands, 64-byte.
// Rows past N read as zero, the code of +0; stores past N are dropped.
int make_map_u8(CUtensorMap* map, const void* ptr, int d, int N, long long BH,
                bool mma_operand = false) {
    EncodeFn enc;
    if (int rc = get_encode(&enc)) return rc;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d),
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                              : (mma_operand ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// FP32 gradient (d, N, B*H) written by TMA stores: 32 x 32 boxes (128-byte
// rows), 128-byte swizzle.  Rows past N are clipped by the copy engine.
int make_map_f32_out(CUtensorMap* map, float* ptr, int d, int N, long long BH) {
    EncodeFn enc;
    if (int rc = get_encode(&enc)) return rc;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 4};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int H, int N, int d, float scale) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;
    const long long tiles = (static_cast<long long>(N) + 127) / 128;
    if (tiles * B * H > (1ll << 31) - 1) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

int check_ptrs(std::initializer_list<const void*> ptrs) {
    for (const void* p : ptrs)
        if (!p) return FA_ERR_INVALID_ARG;
    for (const void* p : ptrs)
        if (!aligned16(p)) return FA_ERR_MISALIGNED;
    return FA_OK;
}

long long n_pad_of(int N) { return (static_cast<long long>(N) + 127) / 128 * 128; }

int launch_rc(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }


// Query heads Hq share Hkv K/V heads (grouped-query attention); Hq = Hkv is
// multi-head attention.
int check_heads(int Hq, int Hkv) {
    if (Hkv < 1 || Hkv > Hq || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int N, int d, int causal, float scale, void* stream) {
    if (int rc = check_ptrs({q, k, v, o, lse})) return rc;
    if (int rc = check_shape(B, Hq, N, d, scale)) return rc;
    if (int rc = check_heads(Hq, Hkv)) return rc;
    unsigned int* status;
    if (int rc = status_ptr(&status)) return rc;
    const long long BH = static_cast<long long>(B) * Hq;
    const long long BHkv = static_cast<long long>(B) * Hkv;
    CUtensorMap tq, tk, tv, to;
    if (int rc = make_map_bf16(&tq, q, d, N, BH)) return rc;
    if (int rc = make_map_bf16(&tk, k, d, N, BHkv)) return rc;
    if (int rc = make_map_bf16(&tv, v, d, N, BHkv)) return rc;
    if (int rc = make_map_bf16(&to, o, d, N, BH)) return rc;
    unsigned int* work;
    int sms;
    if (int rc = work_slot(&work, &sms)) return rc;
    fa::FwdArgs a{&tq, &tk, &tv, &to, lse, B, Hq, N, d, Hkv, causal ? 1 : 0,
                  scale * 1.4426950408889634f, status, g_timeout_ns.load(), work, sms,
                  /*Nk=*/N, /*n_splits=*/1, /*chunk_tiles=*/0, nullptr, nullptr,
                  /*q_scale=*/nullptr, /*k_scale=*/nullptr};
    return launch_rc(fa::launch_fwd_bf16(a, static_cast<cudaStream_t>(stream)));
}

int dkdv_impl(const void* q, const void* k, const void* v, const void* do_,
              const float* delta_ws, const float* lse2_ws, float* dk, float* dv, int B, int Hq,
              int Hkv, int N, int d, int causal, float scale, void* stream) {
    if (int rc = check_ptrs({q, k, v, do_, delta_ws, lse2_ws, dk, dv})) return rc;
    if (int rc = check_shape(B, Hq, N, d, scale)) return rc;
    if (int rc = check_heads(Hq, Hkv)) return rc;
    unsigned int* status;
    if (int rc = status_ptr(&status)) return rc;
    const long long BH = static_cast<long long>(B) * Hq;
    const long long BHkv = static_cast<long long>(B) * Hkv;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv;
    if (int rc = make_map_bf16(&tq, q, d, N, BH)) return rc;
    if (int rc = make_map_bf16(&tk, k, d, N, BHkv)) return rc;
    if (int rc = make_map_bf16(&tv, v, d, N, BHkv)) return rc;
    if (int rc = make_map_bf16(&tdo, do_, d, N, BH)) return rc;
    if (int rc = make_map_f32_out(&tdk, dk, d, N, BHkv)) return rc;
    if (int rc = make_map_f32_out(&tdv, dv, d, N, BHkv)) return rc;
    unsigned int* work;
    int sms;
    if (int rc = work_slot(&work, &sms)) return rc;
    fa::BwdArgs a{&tq, &tk, &tv, &tdo, &tdk, &tdv, delta_ws, lse2_ws, B, Hq, N, d,
                  static_cast<int>(n_pad_of(N)), Hkv, causal ? 1 : 0, scale,
                  scale * 1.4426950408889634f, status, g_timeout_ns.load(), work, sms};
    return launch_rc(fa::launch_bwd_dkdv_bf16(a, static_cast<cudaStream_t>(stream)));
}

// o and lse both null: dQ alone, from delta_ws / lse2_ws as the first step
// wrote them.  Both set: the kernel also does the first step and writes them.
int dq_impl(const void* q, const void* k, const void* v, const void* o, const void* do_,
            const float* lse, float* delta_ws, float* lse2_ws, float* dq, int B, int Hq,
            int Hkv, int N, int d, int causal, float scale, void* stream) {
    if (int rc = check_ptrs({q, k, v, do_, delta_ws, lse2_ws, dq})) return rc;
    if ((o == nullptr) != (lse == nullptr)) return FA_ERR_INVALID_ARG;
    if (o)
        if (int rc = check_ptrs({o, lse})) return rc;
    if (int rc = check_shape(B, Hq, N, d, scale)) return rc;
    if (int rc = check_heads(Hq, Hkv)) return rc;
    unsigned int* status;
    if (int rc = status_ptr(&status)) return rc;
    const long long BH = static_cast<long long>(B) * Hq;
    const long long BHkv = static_cast<long long>(B) * Hkv;
    CUtensorMap tq, tk, tv, tdo, to;
    if (int rc = make_map_bf16(&tq, q, d, N, BH)) return rc;
    if (int rc = make_map_bf16(&tk, k, d, N, BHkv)) return rc;
    if (int rc = make_map_bf16(&tv, v, d, N, BHkv)) return rc;
    if (int rc = make_map_bf16(&tdo, do_, d, N, BH)) return rc;
    if (o)
        if (int rc = make_map_bf16(&to, o, d, N, BH)) return rc;
    unsigned int* work;
    int sms = 0;
    if (int rc = work_slot(&work, &sms)) return rc;
    fa::DqArgs a{&tq, &tk, &tv, &tdo, dq, o, o ? &to : nullptr, lse, delta_ws, lse2_ws, B, Hq, N, d,
                 static_cast<int>(n_pad_of(N)), Hkv, causal ? 1 : 0, scale,
                 scale * 1.4426950408889634f, status, g_timeout_ns.load(), work, sms};
    return launch_rc(fa::launch_bwd_dq_bf16(a, static_cast<cudaStream_t>(stream)));
}

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* do_,
             const float* lse, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int N,
             int d, int causal, float scale, void* workspace, size_t workspace_bytes,
             void* stream);

// Split-KV plan: the key tiles are cut into chunks of chunk_tiles; n_splits
// chunks, none empty.  The query rows of a K/V head's group (g query heads x
// Nq queries, contiguous in memory) form its Q tiles; requested <= 0 lets the
// library choose.  Its choice minimises the time of the busiest SM, modelled
// as waves x (chunk_tiles + 2): waves = ceil(items / SMs) for the (K/V head,
// Q tile, chunk) items, and about two tiles' worth of work per item besides
// its key tiles (Q copy, epilogue, partial store).  A part-filled last wave
// costs a whole one, so the count that fills whole waves wins; on a tie the
// fewer chunks (less to merge).
struct SplitPlan {
    int n_splits;
    int chunk_tiles;
};

long long auto_splits(long long kv_tiles, long long q_items, long long sms) {
    long long best = 1, best_cost = -1;
    for (long long n = 1; n <= kv_tiles && n <= 256; ++n) {
        const long long chunk = (kv_tiles + n - 1) / n;
        const long long used = (kv_tiles + chunk - 1) / chunk;  // chunks actually made
        if (used != n) continue;
        const long long waves = (q_items * n + sms - 1) / sms;
        const long long cost = waves * (chunk + 2);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = n;
        }
    }
    return best;
}

int split_plan(int B, int Hq, int Hkv, int Nq, int Nk, int requested, SplitPlan* out) {
    const long long kv_tiles = (static_cast<long long>(Nk) + 127) / 128;
    const long long group_rows = static_cast<long long>(Hq / Hkv) * Nq;
    const long long q_items = static_cast<long long>(B) * Hkv * ((group_rows + 127) / 128);
    long long want = requested;
    if (want <= 0) {
        unsigned int* unused;
        int sms = 0;
        if (int rc = work_slot(&unused, &sms)) return rc;
        want = auto_splits(kv_tiles, q_items, sms > 0 ? sms : 1);
    }
    if (want < 1) want = 1;
    if (want > kv_tiles) want = kv_tiles;
    const long long chunk = (kv_tiles + want - 1) / want;
    out->chunk_tiles = static_cast<int>(chunk);
    out->n_splits = static_cast<int>((kv_tiles + chunk - 1) / chunk);
    return FA_OK;
}

size_t splitkv_bytes(int B, int Hq, int Nq, int d, int n_splits) {
    const size_t rows = static_cast<size_t>(B) * Hq * Nq * n_splits;
    return rows * static_cast<size_t>(d) * 4 + rows * 4;
}

}  // namespace

extern "C" {

const char* fa_error_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported size or head dimension";
        case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case FA_ERR_CUDA: return "CUDA error";
        case FA_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
        case FA_ERR_NO_MEMORY: return "workspace too small or allocation failed";
        default: return "unknown status";
    }
}

void fa_set_wait_timeout_ns(unsigned long long ns) {
    g_timeout_ns.store(ns < 1000000ull ? 1000000ull : ns);
}

int fa_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_fa_status, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero)) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    if (word & 1u) return FA_ERR_DEVICE_TIMEOUT;
    return word ? FA_ERR_CUDA : FA_OK;  // bit 1: a kernel found its shared memory misplaced
}

int fa_last_device_status(void) { return fa_device_status(0); }

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale, void* stream) {
    return fwd_impl(q, k, v, o, lse, B, H, H, N, d, causal, scale, stream);
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int N, int d, int causal, float scale, void* stream) {
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, stream);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                      int n_splits) {
    if (B < 1 || Hq < 1 || Nq < 1 || Nk < 1 || (d != 64 && d != 128)) return 0;
    if (check_heads(Hq, Hkv) != FA_OK) return 0;
    SplitPlan plan;
    if (split_plan(B, Hq, Hkv, Nq, Nk, n_splits, &plan) != FA_OK) return 0;
    return splitkv_bytes(B, Hq, Nq, d, plan.n_splits);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int Nq, int Nk, int d, float scale, int n_splits,
                   void* workspace, size_t workspace_bytes, void* stream) {
    if (int rc = check_ptrs({q, k, v, o, lse})) return rc;
    if (int rc = check_shape(B, Hq, Nq, d, scale)) return rc;
    if (int rc = check_shape(B, Hkv, Nk, d, scale)) return rc;
    if (int rc = check_heads(Hq, Hkv)) return rc;
    const long long group_rows = static_cast<long long>(Hq / Hkv) * Nq;
    if (group_rows > (1LL << 30)) return FA_ERR_UNSUPPORTED;
    SplitPlan plan;
    if (int rc = split_plan(B, Hq, Hkv, Nq, Nk, n_splits, &plan)) return rc;
    const size_t need = splitkv_bytes(B, Hq, Nq, d, plan.n_splits);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    if (ws) {
        if (!aligned16(ws)) return FA_ERR_MISALIGNED;
        if (workspace_bytes < need) return FA_ERR_NO_MEMORY;
    } else if (cudaMallocAsync(&ws, need, st) != cudaSuccess) {
        return FA_ERR_NO_MEMORY;
    }
    float* o_part = static_cast<float*>(ws);
    float* lse_part = o_part + static_cast<size_t>(B) * Hq * Nq * plan.n_splits * d;
    int rc = FA_OK;
    unsigned int* status;
    unsigned int* work;
    int sms;
    CUtensorMap tq, tk, tv;
    const long long BHkv = static_cast<long long>(B) * Hkv;
    // The g query heads of a K/V head and their Nq queries are contiguous rows
    // of q ([B, Hkv, g, Nq, d]), so the kernel sees each K/V head as one
    // "head" with g * Nq query rows: its Q tiles fill with real rows, and each
    // K/V tile is read once for the whole group.
    const int rows = static_cast<int>(group_rows);
    if ((rc = status_ptr(&status)) == FA_OK && (rc = work_slot(&work, &sms)) == FA_OK &&
        (rc = make_map_bf16(&tq, q, d, rows, BHkv)) == FA_OK &&
        (rc = make_map_bf16(&tk, k, d, Nk, BHkv)) == FA_OK &&
        (rc = make_map_bf16(&tv, v, d, Nk, BHkv)) == FA_OK) {
        // The split kernel stores no O tile: the Q map stands in for O's.
        fa::FwdArgs a{&tq, &tk, &tv, &tq, nullptr, B, Hkv, rows, d, Hkv, 0,
                      scale * 1.4426950408889634f, status, g_timeout_ns.load(), work, sms,
                      Nk, plan.n_splits, plan.chunk_tiles, o_part, lse_part,
                      /*q_scale=*/nullptr, /*k_scale=*/nullptr};
        rc = launch_rc(fa::launch_fwd_splitkv_bf16(a, st));
        if (rc == FA_OK) {
            // Partials and outputs share the row order [B, Hkv, g, Nq] = [B, Hq, Nq].
            fa::CombineArgs c{o_part, lse_part, o, lse, static_cast<int>(BHkv), rows, d,
                              plan.n_splits};
            rc = launch_rc(fa::launch_splitkv_combine(c, st));
        }
    }
    if (!workspace && cudaFreeAsync(ws, st) != cudaSuccess && rc == FA_OK) rc = FA_ERR_CUDA;
    return rc;
}

int fa_fp8_quantize(const void* x, const float* signs, void* codes, float* scales, int BH, int N,
                    int d, void* stream) {
    if (!signs) return FA_ERR_INVALID_ARG;
    if (int rc = check_ptrs({x, codes, scales})) return rc;
    if (int rc = check_shape(1, BH, N, d, 1.f)) return rc;
    fa::Fp8QuantArgs a{};
    for (int i = 0; i < d; ++i) {
        if (signs[i] != 1.f && signs[i] != -1.f) return FA_ERR_INVALID_ARG;
        a.signs.s[i] = signs[i];
    }
    unsigned int* status;
    unsigned int* unused;
    int sms;
    if (int rc = status_ptr(&status)) return rc;
    if (int rc = work_slot(&unused, &sms)) return rc;
    CUtensorMap tx, tc;
    if (int rc = make_map_bf16(&tx, x, d, N, BH)) return rc;
    if (int rc = make_map_u8(&tc, codes, d, N, BH)) return rc;
    a.tm_x = &tx;
    a.tm_codes = &tc;
    a.scales = scales;
    a.BH = BH;
    a.N = N;
    a.d = d;
    a.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    a.status = status;
    a.timeout_ns = g_timeout_ns.load();
    a.num_sms = sms;
    return launch_rc(fa::launch_fp8_rotate_quantize(a, static_cast<cudaStream_t>(stream)));
}

int fa_fwd_fp8(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
               const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
               int causal, float scale, void* stream) {
    if (int rc = check_ptrs({q8, q_scale, k8, k_scale, v, o, lse})) return rc;
    if (int rc = check_shape(B, Hq, N, d, scale)) return rc;
    if (int rc = check_heads(Hq, Hkv)) return rc;
    unsigned int* status;
    if (int rc = status_ptr(&status)) return rc;
    const long long BH = static_cast<long long>(B) * Hq;
    const long long BHkv = static_cast<long long>(B) * Hkv;
    CUtensorMap tq, tk, tv, to;
    if (int rc = make_map_u8(&tq, q8, d, N, BH, true)) return rc;
    if (int rc = make_map_u8(&tk, k8, d, N, BHkv, true)) return rc;
    if (int rc = make_map_bf16(&tv, v, d, N, BHkv)) return rc;
    if (int rc = make_map_bf16(&to, o, d, N, BH)) return rc;
    unsigned int* work;
    int sms;
    if (int rc = work_slot(&work, &sms)) return rc;
    fa::FwdArgs a{&tq, &tk, &tv, &to, lse, B, Hq, N, d, Hkv, causal ? 1 : 0,
                  scale * 1.4426950408889634f, status, g_timeout_ns.load(), work, sms,
                  /*Nk=*/N, /*n_splits=*/1, /*chunk_tiles=*/0, nullptr, nullptr, q_scale, k_scale};
    return launch_rc(fa::launch_fwd_fp8(a, static_cast<cudaStream_t>(stream)));
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
    (void)d;
    if (B < 1 || H < 1 || N < 1) return 0;
    return static_cast<size_t>(2) * static_cast<size_t>(B) * static_cast<size_t>(H) *
           static_cast<size_t>(n_pad_of(N)) * sizeof(float);
}

int fa_bwd_preprocess(const void* o, const void* do_, const float* lse, float* delta_ws,
                      float* lse2_ws, int B, int H, int N, int d, void* stream) {
    if (int rc = check_ptrs({o, do_, lse, delta_ws, lse2_ws})) return rc;
    if (int rc = check_shape(B, H, N, d, 1.f)) return rc;
    fa::BwdPreArgs a{o, do_, lse, delta_ws, lse2_ws, B * H, N, d,
                     static_cast<int>(n_pad_of(N))};
    return launch_rc(fa::launch_bwd_pre_bf16(a, static_cast<cudaStream_t>(stream)));
}

int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* do_,
                const float* delta_ws, const float* lse2_ws, float* dk, float* dv, int B, int H,
                int N, int d, int causal, float scale, void* stream) {
    return dkdv_impl(q, k, v, do_, delta_ws, lse2_ws, dk, dv, B, H, H, N, d, causal, scale,
                     stream);
}

int fa_bwd_dq(const void* q, const void* k, const void* v, const void* do_,
              const float* delta_ws, const float* lse2_ws, float* dq, int B, int H, int N, int d,
              int causal, float scale, void* stream) {
    // The kernel only reads the workspace on this path.
    return dq_impl(q, k, v, nullptr, do_, nullptr, const_cast<float*>(delta_ws),
                   const_cast<float*>(lse2_ws), dq, B, H, H, N, d, causal, scale, stream);
}

int fa_bwd_dq_preprocess(const void* q, const void* k, const void* v, const void* o,
                         const void* do_, const float* lse, float* delta_ws, float* lse2_ws,
                         float* dq, int B, int H, int N, int d, int causal, float scale,
                         void* stream) {
    if (!o || !lse) return FA_ERR_INVALID_ARG;
    return dq_impl(q, k, v, o, do_, lse, delta_ws, lse2_ws, dq, B, H, H, N, d, causal, scale,
                   stream);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* do_,
           const float* lse, float* dq, float* dk, float* dv, int B, int H, int N, int d,
           int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(q, k, v, o, do_, lse, dq, dk, dv, B, H, H, N, d, causal, scale, workspace,
                    workspace_bytes, stream);
}

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* do_,
               const float* lse, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int N,
               int d, int causal, float scale, void* workspace, size_t workspace_bytes,
               void* stream) {
    return bwd_impl(q, k, v, o, do_, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale,
                    workspace, workspace_bytes, stream);
}

int fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
               int H, int N, int d, int causal, float scale, void* stream) {
    if (int rc = check_ptrs({q, k, v, o, lse})) return rc;
    if (int rc = check_shape(B, H, N, d, scale)) return rc;
    if (static_cast<long long>(B) * H > 65535) return FA_ERR_UNSUPPORTED;
    fa::F32Args a{};
    a.q = q; a.k = k; a.v = v; a.out_o = o; a.out_lse = lse;
    a.B = B; a.H = H; a.N = N; a.d = d; a.causal = causal ? 1 : 0; a.scale = scale;
    return launch_rc(fa::launch_fwd_f32(a, static_cast<cudaStream_t>(stream)));
}

int fa_bwd_f32(const float* q, const float* k, const float* v, const float* o, const float* do_,
               const float* lse, float* dq, float* dk, float* dv, int B, int H, int N, int d,
               int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
    if (int rc = check_ptrs({q, k, v, o, do_, lse, dq, dk, dv})) return rc;
    if (int rc = check_shape(B, H, N, d, scale)) return rc;
    if (static_cast<long long>(B) * H > 65535) return FA_ERR_UNSUPPORTED;
    const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    if (ws) {
        if (!aligned16(ws)) return FA_ERR_MISALIGNED;
        if (workspace_bytes < need) return FA_ERR_NO_MEMORY;
    } else if (cudaMallocAsync(&ws, need, s) != cudaSuccess) {
        return FA_ERR_NO_MEMORY;
    }
    fa::F32Args a{};
    a.q = q; a.k = k; a.v = v; a.o = o; a.dO = do_; a.lse = lse;
    a.dq = dq; a.dk = dk; a.dv = dv; a.delta = static_cast<float*>(ws);
    a.B = B; a.H = H; a.N = N; a.d = d; a.causal = causal ? 1 : 0; a.scale = scale;
    int rc = launch_rc(fa::launch_bwd_f32(a, s));
    if (!workspace && cudaFreeAsync(ws, s) != cudaSuccess && rc == FA_OK) rc = FA_ERR_CUDA;
    return rc;
}

int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int* word = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void**>(&word), sizeof(unsigned int), s) != cudaSuccess)
        return FA_ERR_CUDA;
    int rc = FA_OK;
    unsigned int host = 0;
    if (cudaMemsetAsync(word, 0, sizeof(unsigned int), s) != cudaSuccess ||
        fa::launch_wait_timeout_selftest(word, timeout_ns < 1000ull ? 1000ull : timeout_ns, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(&host, word, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        rc = FA_ERR_CUDA;
    cudaFreeAsync(word, s);
    cudaStreamSynchronize(s);
    if (rc != FA_OK) return rc;
    return host ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

}  // extern "C"

namespace {

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* do_,
             const float* lse, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int N,
             int d, int causal, float scale, void* workspace, size_t workspace_bytes,
             void* stream) {
    if (int rc = fa::check_bwd_args(q, k, v, o, do_, lse, dq, dk, dv, B, Hq, N, d, scale))
        return rc;
    if (int rc = check_heads(Hq, Hkv)) return rc;
    const size_t need = fa_bwd_workspace_bytes(B, Hq, N, d);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = workspace;
    if (ws) {
        if (!aligned16(ws)) return FA_ERR_MISALIGNED;
        if (workspace_bytes < need) return FA_ERR_NO_MEMORY;
    } else if (cudaMallocAsync(&ws, need, s) != cudaSuccess) {
        return FA_ERR_NO_MEMORY;
    }
    float* delta = static_cast<float*>(ws);
    float* lse2 = delta + static_cast<size_t>(B) * Hq * n_pad_of(N);
    // dQ with the first step fused writes D and LSE2, then dK/dV reads them.
    int rc = dq_impl(q, k, v, o, do_, lse, delta, lse2, dq, B, Hq, Hkv, N, d, causal, scale,
                     stream);
    if (rc == FA_OK)
        rc = dkdv_impl(q, k, v, do_, delta, lse2, dk, dv, B, Hq, Hkv, N, d, causal, scale, stream);
    if (!workspace && cudaFreeAsync(ws, s) != cudaSuccess && rc == FA_OK) rc = FA_ERR_CUDA;
    return rc;
}

}  // namespace

namespace fa {

int check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* do_,
                   const float* lse, const float* dq, const float* dk, const float* dv, int B,
                   int H, int N, int d, float scale) {
    if (int rc = check_ptrs({q, k, v, o, do_, lse, dq, dk, dv})) return rc;
    return check_shape(B, H, N, d, scale);
}

}  // namespace fa
