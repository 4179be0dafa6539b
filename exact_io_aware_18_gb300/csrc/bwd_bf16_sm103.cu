// bwd_bf16_sm103.cu - attention backward, dK/dV kernel with the dQ atomics,
// BF16 in / FP32 accumulate, tcgen05 + TMEM + TMA on sm_103a.
//
// Method.  The gradient of O = softmax(scale Q K^T) V with the probabilities
// recomputed from the saved LSE instead of read back ("Flash Attention:
// Revolutionizing Transformer Efficiency", section "The Flash Attention
// algorithm", idea 2, recomputation).  Per (b, h), with D_i = dO_i . O_i:
//   P   = exp(scale S - LSE)      dV = P^T dO        dP = dO V^T
//   dS  = P o (dP - D)            dQ = scale dS K    dK = scale dS^T Q
// One CTA owns one 128-key tile j of one (b, h), keeps K_j and V_j in shared
// memory and dK_j, dV_j in TMEM, and loops over the 128-row Q tiles i that
// see those keys (i >= j when causal); the parallelism over key tiles of one
// head is the sequence parallelism of "FlashAttention-2" (technical
// architecture, improvement 2).  Each dQ_i tile is computed on the tensor
// core and added to the FP32 dq buffer with vector atomics.
//
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: K_j, V_j once; per Q tile: Q_i, dO_i tiles and
//               the 128-entry LSE2 / D vectors (bulk copies).
//   warp 1      MMA issuer: S^T = K Q_i^T and dP^T = V dO_i^T (SS), then, once
//               the compute warps have produced P and dS:
//               dV += P^T dO_i (A = P^T from TMEM), dK += dS^T Q_i,
//               dQ_i = dS K (A = dS from shared memory, read M-major).
//   warps 2..5  thread r owns key row r (TMEM lane r): recomputes its row of
//               P^T, forms dS^T, writes P^T (BF16) to TMEM and dS^T (BF16) to
//               shared memory; then, as owners of query rows, read dQ_i out of
//               TMEM and add it to dq; at the end store dK, dV (FP32).
// TMEM columns: S^T [0,128), dP^T / dQ_i [128,256), dV [256,256+d),
// dK [256+d, 256+2d).  Scale is folded into dS before the BF16 rounding.
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

template <int D>
struct BwdCfg {
    static constexpr int BM = 128;  // query rows per Q tile
    static constexpr int BN = 128;  // keys per CTA
    static constexpr int KB = D / 64;
    static constexpr int BOX_BYTES = 128 * 64 * 2;
    static constexpr int TILE_BYTES = KB * BOX_BYTES;
    static constexpr int NSQ = (D == 128) ? 1 : 2;  // Q/dO ring depth
    static constexpr int DS_BYTES = 2 * BOX_BYTES;  // 128 x 128 bf16
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_BYTES;
    static constexpr int OFF_Q = OFF_V + TILE_BYTES;
    static constexpr int OFF_DO = OFF_Q + NSQ * TILE_BYTES;
    static constexpr int OFF_DS = OFF_DO + NSQ * TILE_BYTES;
    static constexpr int OFF_VEC = OFF_DS + DS_BYTES;      // NSQ x (lse2[128], delta[128])
    static constexpr int OFF_BAR = OFF_VEC + NSQ * 1024;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D;
    static constexpr int THREADS = 192;
};

template <int NSQ>
struct BwdBars {
    static constexpr int KV_FULL = 0;
    static constexpr int Q_FULL = 1;
    static constexpr int Q_EMPTY = Q_FULL + NSQ;
    static constexpr int SP_FULL = Q_EMPTY + NSQ;
    static constexpr int DS_FULL = SP_FULL + 1;
    static constexpr int DQ_FULL = DS_FULL + 1;
    static constexpr int DQ_EMPTY = DQ_FULL + 1;
    static constexpr int ACC_FULL = DQ_EMPTY + 1;
    static constexpr int DONE = ACC_FULL + 1;
    static constexpr int COUNT = DONE + 1;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    bwd_dkdv_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const float* __restrict__ delta, const float* __restrict__ lse2,
                         float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
                         int N, int n_pad, int BH, int n_tiles, float scale, float scale_log2,
                         unsigned int* status, unsigned long long timeout_ns) {
    using C = BwdCfg<D>;
    using Bar = BwdBars<C::NSQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_k = s_base + C::OFF_K;
    const uint32_t s_v = s_base + C::OFF_V;
    const uint32_t s_q = s_base + C::OFF_Q;
    const uint32_t s_do = s_base + C::OFF_DO;
    const uint32_t s_ds = s_base + C::OFF_DS;
    const uint32_t s_vec = s_base + C::OFF_VEC;
    const uint32_t s_bar = s_base + C::OFF_BAR;
    auto bar = [&](int slot) -> uint32_t { return s_bar + 8u * static_cast<uint32_t>(slot); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * Bar::COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    // Key tile 0 sees every Q tile under a causal mask: launch it first.
    const long long lin = blockIdx.x + static_cast<long long>(gridDim.x) *
                                           (blockIdx.y + static_cast<long long>(gridDim.y) *
                                                             blockIdx.z);
    const int kt = static_cast<int>(lin / BH);
    const int bh = static_cast<int>(lin % BH);
    const int i0 = CAUSAL ? kt : 0;
    const int n_q = n_tiles - i0;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(Bar::KV_FULL), 1);
        for (int s = 0; s < C::NSQ; ++s) {
            mbar_init(bar(Bar::Q_FULL + s), 1);
            mbar_init(bar(Bar::Q_EMPTY + s), 1);
        }
        mbar_init(bar(Bar::SP_FULL), 1);
        mbar_init(bar(Bar::DS_FULL), 4);
        mbar_init(bar(Bar::DQ_FULL), 1);
        mbar_init(bar(Bar::DQ_EMPTY), 4);
        mbar_init(bar(Bar::ACC_FULL), 1);
        mbar_init(bar(Bar::DONE), 1);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_do);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const WaitCtx wc{status, timeout_ns, abort_flag};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(Bar::KV_FULL), 2 * C::TILE_BYTES);
            for (int kb = 0; kb < C::KB; ++kb) {
                tma_load_3d(s_k + kb * C::BOX_BYTES, &tm_k, bar(Bar::KV_FULL), kb * 64,
                            kt * C::BN, bh);
                tma_load_3d(s_v + kb * C::BOX_BYTES, &tm_v, bar(Bar::KV_FULL), kb * 64,
                            kt * C::BN, bh);
            }
            int issued = 0;
            for (int t = 0; t < n_q; ++t) {
                const int st = t % C::NSQ;
                const int use = t / C::NSQ;
                if (use > 0 && !mbar_wait(bar(Bar::Q_EMPTY + st), (use - 1) & 1, wc)) break;
                const int i = i0 + t;
                const uint32_t fb = bar(Bar::Q_FULL + st);
                mbar_arrive_expect_tx(fb, 2 * C::TILE_BYTES + 1024);
                for (int kb = 0; kb < C::KB; ++kb) {
                    tma_load_3d(s_q + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_q, fb,
                                kb * 64, i * C::BM, bh);
                    tma_load_3d(s_do + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_do, fb,
                                kb * 64, i * C::BM, bh);
                }
                const long long voff = static_cast<long long>(bh) * n_pad + i * C::BM;
                bulk_load(s_vec + st * 1024, lse2 + voff, 512, fb);
                bulk_load(s_vec + st * 1024 + 512, delta + voff, 512, fb);
                issued = t + 1;
            }
            mbar_wait_drain(bar(Bar::KV_FULL), 0, timeout_ns);
            for (int t = (issued > C::NSQ ? issued - C::NSQ : 0); t < issued; ++t)
                mbar_wait_drain(bar(Bar::Q_FULL + t % C::NSQ), (t / C::NSQ) & 1, timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_sp = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
            constexpr uint32_t id_kv = idesc_bf16(128, D, 0, 1);    // dV, dK: B MN-major
            constexpr uint32_t id_q = idesc_bf16(128, D, 1, 1);     // dQ: A and B MN-major
            bool ok = mbar_wait(bar(Bar::KV_FULL), 0, wc);
            for (int t = 0; t < n_q && ok; ++t) {
                const int st = t % C::NSQ;
                const uint32_t q_tile = s_q + st * C::TILE_BYTES;
                const uint32_t do_tile = s_do + st * C::TILE_BYTES;
                ok = mbar_wait(bar(Bar::Q_FULL + st), (t / C::NSQ) & 1, wc);
                if (ok && t > 0) ok = mbar_wait(bar(Bar::DQ_EMPTY), (t - 1) & 1, wc);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                    mma_ss(tmem + C::COL_S, smem_desc_sw128(s_k + koff, 16, 1024),
                           smem_desc_sw128(q_tile + koff, 16, 1024), id_sp, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                    mma_ss(tmem + C::COL_DP, smem_desc_sw128(s_v + koff, 16, 1024),
                           smem_desc_sw128(do_tile + koff, 16, 1024), id_sp, kk > 0);
                }
                tc_commit(bar(Bar::SP_FULL));
                ok = mbar_wait(bar(Bar::DS_FULL), t & 1, wc);
                if (!ok) break;
                tc_fence_after();
                const uint32_t acc = (t > 0) ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)  // dV += P^T dO_i
                    mma_ts(tmem + C::COL_DV, tmem + C::COL_S + kk * 8,
                           smem_desc_sw128(do_tile + kk * 2048, C::BOX_BYTES, 1024), id_kv,
                           acc | (kk > 0));
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk)  // dK += dS^T Q_i
                    mma_ss(tmem + C::COL_DK,
                           smem_desc_sw128(s_ds + (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32, 16,
                                           1024),
                           smem_desc_sw128(q_tile + kk * 2048, C::BOX_BYTES, 1024), id_kv,
                           acc | (kk > 0));
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)  // dQ_i = dS K
                    mma_ss(tmem + C::COL_DP,
                           smem_desc_sw128(s_ds + kk * 2048, C::BOX_BYTES, 1024),
                           smem_desc_sw128(s_k + kk * 2048, C::BOX_BYTES, 1024), id_q, kk > 0);
                tc_commit(bar(Bar::Q_EMPTY + st));
                tc_commit(bar(Bar::DQ_FULL));
            }
            if (ok) tc_commit(bar(Bar::ACC_FULL));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute
        const int wq = warp & 3;
        const int r = wq * 32 + lane;            // key row (then query row for dQ)
        const int kglob = kt * C::BN + r;        // key index inside the head
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float* vec_base = reinterpret_cast<const float*>(smem + C::OFF_VEC);
        uint8_t* ds_rows = smem + C::OFF_DS;
        const long long head_row0 = static_cast<long long>(bh) * N;
        bool ok = true;
        for (int t = 0; t < n_q; ++t) {
            const int st = t % C::NSQ;
            const int i = i0 + t;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::SP_FULL), t & 1, wc) &&
                                             mbar_wait(bar(Bar::Q_FULL + st),
                                                       (t / C::NSQ) & 1, wc));
            if (!ok) break;
            tc_fence_after();
            const float* l2v = vec_base + st * 256;
            const float* dlt = l2v + 128;
            const bool diag = CAUSAL && i == kt;
            const bool key_pad = kglob >= N;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t sr[32], dr[32];
                tmem_ld32(t_lane + C::COL_S + ch * 32, sr);
                tmem_ld32(t_lane + C::COL_DP + ch * 32, dr);
                uint32_t pk[16];
                uint32_t dk2[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float pe[2], de[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = ch * 32 + 2 * e + h;  // query column in the tile
                        float p = ex2_approx(
                            fmaf(__uint_as_float(sr[2 * e + h]), scale_log2, -l2v[c]));
                        if (key_pad || (diag && i * C::BM + c < kglob)) p = 0.f;
                        pe[h] = p;
                        de[h] = p * (__uint_as_float(dr[2 * e + h]) - dlt[c]) * scale;
                    }
                    pk[e] = pack_bf16x2(pe[0], pe[1]);
                    dk2[e] = pack_bf16x2(de[0], de[1]);
                }
                tmem_st16(t_lane + C::COL_S + ch * 16, pk);
                // dS^T row r, queries ch*32 .. ch*32+31: four 16-byte chunks.
                const int box = ch >> 1;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int chunk = ((ch & 1) * 4 + u) ^ (r & 7);
                    *reinterpret_cast<uint4*>(ds_rows + box * C::BOX_BYTES + r * 128 +
                                              chunk * 16) =
                        make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
                }
            }
            tmem_st_wait();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::DS_FULL));

            // dQ_i tile: lane r now owns query row r of the tile.
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::DQ_FULL), t & 1, wc));
            if (!ok) break;
            tc_fence_after();
            const int qglob = i * C::BM + r;
            float4* dq_row = reinterpret_cast<float4*>(dq + (head_row0 + qglob) * D);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t qr[32];
                tmem_ld32(t_lane + C::COL_DP + ch * 32, qr);
                if (qglob < N) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        atomicAdd(dq_row + ch * 8 + u,
                                  make_float4(__uint_as_float(qr[4 * u]),
                                              __uint_as_float(qr[4 * u + 1]),
                                              __uint_as_float(qr[4 * u + 2]),
                                              __uint_as_float(qr[4 * u + 3])));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::DQ_EMPTY));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::ACC_FULL), 0, wc));
        if (ok) {
            tc_fence_after();
            float4* dv_row = reinterpret_cast<float4*>(dv + (head_row0 + kglob) * D);
            float4* dk_row = reinterpret_cast<float4*>(dk + (head_row0 + kglob) * D);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t a[32], b[32];
                tmem_ld32(t_lane + C::COL_DV + ch * 32, a);
                tmem_ld32(t_lane + C::COL_DK + ch * 32, b);
                if (kglob < N) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        dv_row[ch * 8 + u] =
                            make_float4(__uint_as_float(a[4 * u]), __uint_as_float(a[4 * u + 1]),
                                        __uint_as_float(a[4 * u + 2]),
                                        __uint_as_float(a[4 * u + 3]));
                        dk_row[ch * 8 + u] =
                            make_float4(__uint_as_float(b[4 * u]), __uint_as_float(b[4 * u + 1]),
                                        __uint_as_float(b[4 * u + 2]),
                                        __uint_as_float(b[4 * u + 3]));
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) {
            tc_commit(bar(Bar::DONE));
            mbar_wait_drain(bar(Bar::DONE), 0, timeout_ns);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t stream) {
    using C = BwdCfg<D>;
    auto kern = bwd_dkdv_bf16_kernel<D, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.N + C::BN - 1) / C::BN;
    dim3 grid(n_tiles, a.H, a.B);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(
        *a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, a.delta, a.lse2, a.dq, a.dk, a.dv, a.N, a.n_pad,
        a.B * a.H, n_tiles, a.scale, a.scale_log2, a.status, a.timeout_ns);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
    return a.causal ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
}

}  // namespace fa
