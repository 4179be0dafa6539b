// bwd_bf16_sm103.cu - attention backward, dK/dV kernel, BF16 in / FP32
// accumulate, tcgen05 + TMEM + TMA on sm_103a.
//
// Method.  The gradient of O = softmax(scale Q K^T) V with the probabilities
// recomputed from the saved LSE instead of read back ("Flash Attention:
// Revolutionizing Transformer Efficiency", section "The Flash Attention
// algorithm", idea 2, recomputation).  Per (b, h), with D_i = dO_i . O_i:
//   P   = exp(scale S - LSE)      dV = P^T dO        dP = dO V^T
//   dS  = P o (dP - D)            dK = scale dS^T Q  (dQ: bwd_dq_sm103.cu)
// One CTA owns one 128-key tile j of one (b, h), keeps K_j and V_j in shared
// memory and dK_j, dV_j in TMEM, and loops over the 128-row Q tiles i that
// see those keys (i >= j when causal); the parallelism over key tiles of one
// head is the sequence parallelism of "FlashAttention-2" (technical
// architecture, improvement 2).  dQ is left to a second kernel that loops
// over key tiles per Q tile, so nothing here is reduced across CTAs.
//
// Roles (352 threads, one CTA per SM):
//   warp 0      TMA producer: K_j, V_j once; per Q tile, into a two-deep ring
//               of [Q_i | dO_i] stages plus the 128-entry LSE2 / D vectors.
//   warps 1, 10 two MMA issuers (one thread each).  A single thread issues a
//               128 x 128 x 16 tcgen05.mma about as fast as the tensor pipe
//               runs it, so every barrier check in between would leave the
//               pipe idle; with two issuers one keeps the pipe fed while the
//               other waits.  Each issuer overwrites only TMEM it alone reads,
//               after those reads in its own issue order:
//                 issuer A: dV += P^T_t dO_t (A = P^T in TMEM, after P_FULL),
//                           then S^T_t+1 = K Q_t+1^T over P^T_t;
//                 issuer B: dK += dS^T_t Q_t (A = dS^T in TMEM, after DS_FULL),
//                           then dP^T_t+1 = V dO_t+1^T over dS^T_t.
//               So S^T and dP^T of the next tile run while the P and dS math
//               of this one does.  A stage is free once both issuers commit.
//   warps 2..9  thread (r, h) owns key row r (TMEM lane r) and column half h
//               (warps 2-5: h = 0, warps 6-9: h = 1).  Phase P: 64 entries of
//               the P^T row = exp2(S^T * scale*log2e - LSE2), kept in
//               registers and written back as BF16 into the first 32 of its
//               own 64 S^T columns.  Phase dS: dS^T = P o (dP^T - D), BF16,
//               likewise into its own dP^T columns (scale is applied to dK
//               once, when it leaves TMEM).  At the end: dK, dV rows out of
//               TMEM into swizzled shared-memory boxes, then to global memory
//               (FP32) by TMA stores of whole 128-byte rows.
// TMEM columns: S^T [0,128) (P^T halves at [0,32) and [64,96)),
// dP^T [128,256) (dS^T halves at [128,160) and [192,224)), dV [256,256+d),
// dK [256+d, 256+2d).  Eleven warps cap a thread at 168 registers (the
// register file is split among the four SM sub-partitions, three warps on
// three of them).  All waits are bounded (see sm103_primitives.cuh).
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kMaxDynSmem = 232448;  // 227 KB opt-in limit per block

template <int D>
struct BwdCfg {
    static constexpr int BM = 128;  // query rows per Q tile
    static constexpr int BN = 128;  // keys per CTA
    static constexpr int KB = D / 64;
    static constexpr int BOX_BYTES = 128 * 64 * 2;      // 128 x 64 bf16
    static constexpr int TILE_BYTES = KB * BOX_BYTES;    // 128 x D bf16
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // [Q | dO]
    static constexpr int NSQ = 2;                        // stage ring depth
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_BYTES;
    static constexpr int OFF_STAGE = OFF_V + TILE_BYTES;
    static constexpr int OFF_VEC = OFF_STAGE + NSQ * STAGE_BYTES;  // NSQ x (lse2, delta)
    static constexpr int OFF_BAR = OFF_VEC + NSQ * 1024;
    static constexpr int BAR_BYTES = 256;
    static constexpr int LAYOUT_BYTES = OFF_BAR + BAR_BYTES;
    static constexpr int SMEM_BYTES =
        (LAYOUT_BYTES + 1024 <= kMaxDynSmem) ? LAYOUT_BYTES + 1024 : kMaxDynSmem;
    static_assert(LAYOUT_BYTES <= kMaxDynSmem, "backward tiles do not fit in shared memory");
    // The epilogue stages FP32 dV and dK (2 x 8 warps x d/64 boxes of 4 KB)
    // over K, V and the stage ring, which start at offset 0 and are contiguous.
    static_assert(OFF_K == 0 && 2 * 8 * (D / 64) * 4096 <= OFF_VEC,
                  "dK/dV staging does not fit over the tiles");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D;
    static constexpr int THREADS = 352;
    static constexpr int COMPUTE_WARPS = 8;
};

template <int NSQ>
struct BwdBars {
    static constexpr int KV_FULL = 0;
    static constexpr int Q_FULL = 1;
    static constexpr int Q_EMPTY = Q_FULL + NSQ;
    static constexpr int S_FULL = Q_EMPTY + NSQ;
    static constexpr int DP_FULL = S_FULL + 1;
    static constexpr int P_FULL = DP_FULL + 1;
    static constexpr int DS_FULL = P_FULL + 1;
    static constexpr int ACC_FULL = DS_FULL + 1;
    static constexpr int DONE = ACC_FULL + 1;
    static constexpr int COUNT = DONE + 1;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(352, 1)
    bwd_dkdv_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk,
                         const __grid_constant__ CUtensorMap tm_dv,
                         const float* __restrict__ delta, const float* __restrict__ lse2,
                         int N, int n_pad, int BHkv, int Hkv, int n_rep, int n_tiles,
                         int group, float scale, float scale_log2, unsigned int* status,
                         unsigned long long timeout_ns) {
    using C = BwdCfg<D>;
    using Bar = BwdBars<C::NSQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    if (smem + C::LAYOUT_BYTES > smem_raw + C::SMEM_BYTES) {
        // The dynamic shared memory did not start on a 1024-byte boundary and
        // the tiles do not fit after aligning: report it and do nothing.
        if (threadIdx.x == 0) atomicOr(status, kStatusSmemLayout);
        return;
    }
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_k = s_base + C::OFF_K;
    const uint32_t s_v = s_base + C::OFF_V;
    const uint32_t s_stage = s_base + C::OFF_STAGE;
    const uint32_t s_vec = s_base + C::OFF_VEC;
    const uint32_t s_bar = s_base + C::OFF_BAR;
    auto bar = [&](int slot) -> uint32_t { return s_bar + 8u * static_cast<uint32_t>(slot); };
    auto q_of = [&](int st) -> uint32_t { return s_stage + st * C::STAGE_BYTES; };
    auto do_of = [&](int st) -> uint32_t { return s_stage + st * C::STAGE_BYTES + C::TILE_BYTES; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * Bar::COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    // Key tile 0 sees every Q tile under a causal mask: heavy tiles first,
    // a few heads at a time so their Q and dO stay in L2.
    const long long lin = blockIdx.x + static_cast<long long>(gridDim.x) *
                                           (blockIdx.y + static_cast<long long>(gridDim.y) *
                                                             blockIdx.z);
    const TileHead th = grouped_order(lin, BHkv, n_tiles, group, false);
    const int kt = th.tile;
    const int bkv = th.head;  // K/V head (b * Hkv + j)
    const int i0 = CAUSAL ? kt : 0;
    const int n_q = n_tiles - i0;
    // Step t covers query head r = t / n_q of this K/V head's group (the
    // n_rep query heads b * Hq + j * n_rep + r, Hq = n_rep * Hkv) and its Q
    // tile i = i0 + t % n_q; with n_rep = 1 this is plain multi-head attention.
    const int n_steps = n_rep * n_q;
    const int bhq0 = (bkv / Hkv) * (Hkv * n_rep) + (bkv % Hkv) * n_rep;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(Bar::KV_FULL), 1);
        for (int s = 0; s < C::NSQ; ++s) {
            mbar_init(bar(Bar::Q_FULL + s), 1);
            mbar_init(bar(Bar::Q_EMPTY + s), 2);  // one commit per issuer
        }
        mbar_init(bar(Bar::S_FULL), 1);
        mbar_init(bar(Bar::DP_FULL), 1);
        mbar_init(bar(Bar::P_FULL), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::DS_FULL), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::ACC_FULL), 2);
        mbar_init(bar(Bar::DONE), 2);
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
            auto load_tile = [&](int t) {
                const int st = t % C::NSQ;
                const int i = i0 + t % n_q;
                const int bh = bhq0 + t / n_q;  // query head
                const uint32_t fb = bar(Bar::Q_FULL + st);
                mbar_arrive_expect_tx(fb, C::STAGE_BYTES + 1024);
                for (int kb = 0; kb < C::KB; ++kb) {
                    tma_load_3d(q_of(st) + kb * C::BOX_BYTES, &tm_q, fb, kb * 64, i * C::BM, bh);
                    tma_load_3d(do_of(st) + kb * C::BOX_BYTES, &tm_do, fb, kb * 64, i * C::BM,
                                bh);
                }
                const long long voff = static_cast<long long>(bh) * n_pad + i * C::BM;
                bulk_load(s_vec + st * 1024, lse2 + voff, 512, fb);
                bulk_load(s_vec + st * 1024 + 512, delta + voff, 512, fb);
            };
            mbar_arrive_expect_tx(bar(Bar::KV_FULL), 2 * C::TILE_BYTES);
            for (int kb = 0; kb < C::KB; ++kb) {
                tma_load_3d(s_k + kb * C::BOX_BYTES, &tm_k, bar(Bar::KV_FULL), kb * 64,
                            kt * C::BN, bkv);
                tma_load_3d(s_v + kb * C::BOX_BYTES, &tm_v, bar(Bar::KV_FULL), kb * 64,
                            kt * C::BN, bkv);
            }
            int issued = 0;
            for (; issued < n_steps; ++issued) {
                const int use = issued / C::NSQ;
                if (use > 0 &&
                    !mbar_wait(bar(Bar::Q_EMPTY + issued % C::NSQ), (use - 1) & 1, wc))
                    break;
                load_tile(issued);
            }
            mbar_wait_drain(bar(Bar::KV_FULL), 0, timeout_ns);
            for (int t = (issued > C::NSQ ? issued - C::NSQ : 0); t < issued; ++t)
                mbar_wait_drain(bar(Bar::Q_FULL + t % C::NSQ), (t / C::NSQ) & 1, timeout_ns);
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------------------ MMA issuers
        if (lane == 0) {
            constexpr uint32_t id_sp = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
            constexpr uint32_t id_kv = idesc_bf16(128, D, 0, 1);    // dV, dK: B MN-major
            const bool issuer_a = (warp == 1);
            // Base descriptors; each MMA below only moves the start address.
            const uint64_t d_k = smem_desc_sw128(s_k, 16, 1024);                // A of S^T
            const uint64_t d_v = smem_desc_sw128(s_v, 16, 1024);                // A of dP^T
            // Stage 0 descriptors; stage st sits st * STAGE_BYTES further on.
            // issuer A: Q (K-major, B of S^T) and dO (MN-major, B of dV);
            // issuer B: dO (K-major, B of dP^T) and Q (MN-major, B of dK).
            const uint64_t d_kmaj0 = smem_desc_sw128(issuer_a ? q_of(0) : do_of(0), 16, 1024);
            const uint64_t d_mn0 = smem_desc_sw128(issuer_a ? do_of(0) : q_of(0), C::BOX_BYTES, 1024);
            const uint64_t d_first = issuer_a ? d_k : d_v;
            const uint32_t c_first = issuer_a ? C::COL_S : C::COL_DP;   // S^T or dP^T
            const uint32_t c_acc = issuer_a ? C::COL_DV : C::COL_DK;    // dV or dK
            const uint32_t c_a = issuer_a ? C::COL_S : C::COL_DP;       // P^T or dS^T
            const int ready_bar = issuer_a ? Bar::P_FULL : Bar::DS_FULL;
            const int full_bar = issuer_a ? Bar::S_FULL : Bar::DP_FULL;
            // First GEMM of tile t: S^T_t = K Q_t^T (A) or dP^T_t = V dO_t^T (B).
            auto issue_first = [&](int t) -> bool {
                const int st = t % C::NSQ;
                if (!mbar_wait(bar(Bar::Q_FULL + st), (t / C::NSQ) & 1, wc)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                    mma_ss(tmem + c_first, desc_advance(d_first, koff),
                           desc_advance(d_kmaj0, st * C::STAGE_BYTES + koff), id_sp, kk > 0);
                }
                tc_commit(bar(full_bar));
                return true;
            };
            bool ok = mbar_wait(bar(Bar::KV_FULL), 0, wc) && issue_first(0);
            for (int t = 0; t < n_steps && ok; ++t) {
                const int st = t % C::NSQ;
                ok = mbar_wait(bar(ready_bar), t & 1, wc);
                if (!ok) break;
                tc_fence_after();
                // dV += P^T_t dO_t (A) or dK += dS^T_t Q_t (B); the BF16 halves
                // of P^T / dS^T (queries 0-63, 64-127) sit at columns [0,32) and
                // [64,96) of their fp32 region.
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk) {
                    const uint32_t acol = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
                    mma_ts(tmem + c_acc, tmem + c_a + acol, desc_advance(d_mn0, st * C::STAGE_BYTES + kk * 2048),
                           id_kv, (t > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(Bar::Q_EMPTY + st));  // this issuer no longer reads stage t
                if (t + 1 < n_steps) ok = issue_first(t + 1);
            }
            if (ok) tc_commit(bar(Bar::ACC_FULL));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ P / dS
        const int wq = warp & 3;
        const int h = (warp - 2) >> 2;       // column half
        const int r = wq * 32 + lane;        // key row
        const int kglob = kt * C::BN + r;    // key index inside the head
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float* vec_base = reinterpret_cast<const float*>(smem + C::OFF_VEC);
        const bool key_pad = kglob >= N;
        bool ok = true;
        for (int t = 0; t < n_steps; ++t) {
            const int st = t % C::NSQ;
            const int i = i0 + t % n_q;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::S_FULL), t & 1, wc) &&
                                             mbar_wait(bar(Bar::Q_FULL + st),
                                                       (t / C::NSQ) & 1, wc));
            if (!ok) break;
            tc_fence_after();
            const float* l2v = vec_base + st * 256 + 64 * h;
            const float* dlt = vec_base + st * 256 + 128 + 64 * h;
            // Phase P: entries [64h, 64h+64) of this key's row of P^T.
            float p[64];
            {
                uint32_t sr[64];
                tmem_ld64(t_lane + C::COL_S + 64 * h, sr);
                const int q0 = i * C::BM + 64 * h;  // query index of entry 0
                if (key_pad || (CAUSAL && i == kt)) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const float x =
                            ex2_approx(fmaf(__uint_as_float(sr[c]), scale_log2, -l2v[c]));
                        p[c] = (key_pad || q0 + c < kglob) ? 0.f : x;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        p[c] = ex2_approx(fmaf(__uint_as_float(sr[c]), scale_log2, -l2v[c]));
                }
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
                tmem_st32(t_lane + C::COL_S + 64 * h, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::P_FULL));

            // Phase dS: dS^T = P o (dP^T - D) * scale, BF16, over its dP^T columns.
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::DP_FULL), t & 1, wc));
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t dr[64];
                tmem_ld64(t_lane + C::COL_DP + 64 * h, dr);
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int c = 2 * e;
                    w[e] = pack_bf16x2(p[c] * (__uint_as_float(dr[c]) - dlt[c]),
                                       p[c + 1] * (__uint_as_float(dr[c + 1]) - dlt[c + 1]));
                }
                tmem_st32(t_lane + C::COL_DP + 64 * h, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::DS_FULL));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::ACC_FULL), 0, wc));
        if (ok) {
            // Every MMA has completed, so K, V and the [Q | dO] ring hold the
            // staging boxes: this warp's 32 rows x d/2 columns of dV, then of
            // dK, as d/64 boxes of 32 x 32 each, stored by TMA in whole
            // 128-byte rows.
            tc_fence_after();
            constexpr uint32_t kHalfBytes = 8 * (D / 64) * 4096;  // all of dV
            const uint32_t stg = s_k + static_cast<uint32_t>((warp - 2) * (D / 64) * 4096);
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch) {
                uint32_t a[32];
                tmem_ld32(t_lane + C::COL_DV + (D / 2) * h + ch * 32, a);
                st_row_sw128_f32(stg + ch * 4096, lane, a, 1.f);
                tmem_ld32(t_lane + C::COL_DK + (D / 2) * h + ch * 32, a);
                st_row_sw128_f32(stg + kHalfBytes + ch * 4096, lane, a, scale);
            }
            fence_async_smem();
            __syncwarp();
            const int row0 = kt * C::BN + wq * 32;
            if (lane == 0 && row0 < N) {
#pragma unroll
                for (int ch = 0; ch < D / 64; ++ch) {
                    tma_store_3d(&tm_dv, stg + ch * 4096, (D / 2) * h + ch * 32, row0, bkv);
                    tma_store_3d(&tm_dk, stg + kHalfBytes + ch * 4096, (D / 2) * h + ch * 32,
                                 row0, bkv);
                }
                bulk_commit();
                bulk_wait_read_all();  // the boxes stay in place until read
            }
            __syncwarp();
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (warp == 10 && lane == 0) tc_commit(bar(Bar::DONE));
    if (warp == 1) {
        if (lane == 0) {
            tc_commit(bar(Bar::DONE));  // both issuers' MMAs have completed
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
    // Enough heads per group that a group fills about one wave of CTAs.
    int group = 128 / n_tiles;
    if (group < 1) group = 1;
    dim3 grid(n_tiles, a.Hkv, a.B);  // one CTA per key tile of each K/V head
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(
        *a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dk, *a.tm_dv, a.delta, a.lse2, a.N, a.n_pad,
        a.B * a.Hkv, a.Hkv, a.H / a.Hkv, n_tiles, group, a.scale, a.scale_log2, a.status,
        a.timeout_ns);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
    return a.causal ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
}

}  // namespace fa
