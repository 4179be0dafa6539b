// bwd_dq_sm103.cu - attention backward, dQ kernel, BF16 in / FP32 out,
// tcgen05 + TMEM + TMA on sm_103a.
//
// Method.  dQ = scale dS K with dS = P o (dP - D), P = exp(scale Q K^T - LSE)
// recomputed from the saved LSE ("Flash Attention: Revolutionizing
// Transformer Efficiency", section "The Flash Attention algorithm", idea 2,
// recomputation) and dP = dO V^T.  One CTA owns one 128-row Q tile of one
// (b, h) and loops over the key tiles it sees (j <= i when causal), exactly
// like the forward's loop order ("FlashAttention scaling, multi-GPU training
// and weight quantization", section 1): the dQ tile accumulates in TMEM and is
// written once, so the result does not depend on the order in which CTAs run
// (no atomics; "FlashAttention-2" stresses a deterministic exact result).
//
// Roles (384 threads, one CTA per SM):
//   warp 0      TMA producer: (given O) the O tile into the third K stage
//               first, then Q_i and dO_i once, then K_j into a three-deep ring
//               (K_j is read until the dQ MMA of tile j); K_2 waits until the
//               math warps have read O.
//   warp 11     TMA producer: V_j into a two-deep ring (read only by dP_j).
//               The two rings free at different times, so each has its own
//               thread, and each thread its own warp: two lanes of one warp
//               that both spin on barriers share one instruction stream.
//   warps 1, 10 two MMA issuers, so that one keeps the pipe fed while the
//               other waits (issuer B a whole warp with one elected lane;
//               issuer A likewise without a causal mask, lane 0 alone with
//               one, as measured fastest).  Issuer A: S_0, S_1, then
//               per key tile j: dQ += dS_j K_j (A = dS_j in TMEM, after
//               DS_FULL) and S_j+2 = Q K_j+2^T over dS_j.  Issuer B: (given O)
//               D = diag(dO O^T) into the dQ columns, dP_0, then
//               dP_j+1 = dO V_j+1^T as soon as the math warps hold dP_j in
//               registers.  S is double buffered and dP is released early, so
//               both operands of tile j+1 are ready when the math of tile j
//               ends.
//   warps 2..9  thread (r, h) owns query row r (TMEM lane r) and key half h.
//               Given O and LSE, the backward's first step for their rows
//               comes first: D_r = sum_c dO_rc O_rc is the diagonal of dO O^T,
//               which issuer B computes on the tensor core into the dQ
//               columns before any dP (O arrives by TMA in the third K stage);
//               each thread reads its diagonal entry and writes D and
//               LSE2_r = LSE_r log2 e out for the dK/dV kernel.  Else they
//               read both.
//               Per key tile:
//               P' = exp2(S * scale*log2e - LSE2_r + log2 scale) = scale P,
//               dS' = P' o (dP - D_r) = scale dS, BF16, written over the first
//               32 of its own 64 S columns.  At the end: the dQ row half out
//               of TMEM into swizzled shared-memory boxes, then to global
//               memory (FP32) by TMA stores of whole 128-byte rows.
// TMEM columns: S buffers [0,128) and [128,256), dP [256,384), dQ [384,384+d)
// (dO O^T takes [384,512) before the first dQ product).
// All waits are bounded (see sm103_primitives.cuh).
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kMaxDynSmem = 232448;  // 227 KB opt-in limit per block

template <int D>
struct DqCfg {
    static constexpr int BM = 128;  // query rows per CTA
    static constexpr int BN = 128;  // keys per tile
    static constexpr int KB = D / 64;
    static constexpr int BOX_BYTES = 128 * 64 * 2;
    static constexpr int TILE_BYTES = KB * BOX_BYTES;
    static constexpr int NSK = 3;  // K ring depth
    static constexpr int NSV = 2;  // V ring depth
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + TILE_BYTES;
    static constexpr int OFF_K = OFF_DO + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + NSV * TILE_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int LAYOUT_BYTES = OFF_BAR + BAR_BYTES;
    static constexpr int SMEM_BYTES =
        (LAYOUT_BYTES + 1024 <= kMaxDynSmem) ? LAYOUT_BYTES + 1024 : kMaxDynSmem;
    static_assert(LAYOUT_BYTES <= kMaxDynSmem, "dQ tiles do not fit in shared memory");
    // The epilogue stages the FP32 dQ tile (8 warps x d/64 boxes of 4 KB) over Q and dO.
    static_assert(8 * (D / 64) * 4096 <= 2 * TILE_BYTES && OFF_DO == OFF_Q + TILE_BYTES,
                  "dQ staging does not fit over Q and dO");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_DP = 256, COL_DQ = 384;
    static constexpr int THREADS = 384;
    static constexpr int COMPUTE_WARPS = 8;
};

template <int NSK, int NSV>
struct DqBars {
    static constexpr int QD_FULL = 0;
    static constexpr int K_FULL = 1;
    static constexpr int K_EMPTY = K_FULL + NSK;
    static constexpr int V_FULL = K_EMPTY + NSK;
    static constexpr int V_EMPTY = V_FULL + NSV;
    static constexpr int S_FULL = V_EMPTY + NSV;  // 2
    static constexpr int DP_FULL = S_FULL + 2;
    static constexpr int DP_EMPTY = DP_FULL + 1;
    // One dS barrier per S buffer.  S_j+2 is issued right after dQ_j, so the
    // math warps may finish key tiles j + 1 and j + 2 before issuer A looks
    // for dS_j+1; on a single barrier that second phase would hide the first
    // from A's parity wait.  Per buffer, they can be at most one phase ahead.
    static constexpr int DS_FULL = DP_EMPTY + 1;  // 2
    static constexpr int O_FULL = DS_FULL + 2;
    static constexpr int O_FREE = O_FULL + 1;
    static constexpr int D_FULL = O_FREE + 1;
    static constexpr int DQ_DONE = D_FULL + 1;
    static constexpr int DONE = DQ_DONE + 1;
    static constexpr int COUNT = DONE + 1;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq,
                       const __grid_constant__ CUtensorMap tm_o, int fused,
                       const float* __restrict__ lse,
                       float* __restrict__ delta, float* __restrict__ lse2, int N, int n_pad, int BH,
                       int Hq, int n_rep, int n_tiles, int group,
                       float scale, float scale_log2, unsigned int* status,
                       unsigned long long timeout_ns) {
    using C = DqCfg<D>;
    using Bar = DqBars<C::NSK, C::NSV>;
    static_assert(8 * Bar::COUNT + 8 <= C::BAR_BYTES, "barrier area");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    if (smem + C::LAYOUT_BYTES > smem_raw + C::SMEM_BYTES) {
        if (threadIdx.x == 0) atomicOr(status, kStatusSmemLayout);
        return;
    }
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + C::OFF_Q;
    const uint32_t s_do = s_base + C::OFF_DO;
    const uint32_t s_k = s_base + C::OFF_K;
    const uint32_t s_v = s_base + C::OFF_V;
    const uint32_t s_bar = s_base + C::OFF_BAR;
    auto bar = [&](int slot) -> uint32_t { return s_bar + 8u * static_cast<uint32_t>(slot); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * Bar::COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    // Heavy Q tiles first (the last Q tile sees the most keys under a causal
    // mask), a few heads at a time so that their K and V stay in L2.
    const long long lin = blockIdx.x + static_cast<long long>(gridDim.x) *
                                           (blockIdx.y + static_cast<long long>(gridDim.y) *
                                                             blockIdx.z);
    const TileHead th = grouped_order(lin, BH, n_tiles, group, true);
    const int qt = th.tile;
    const int bh = th.head;
    // K/V head of query head bh: its group's head (b * Hkv + h / n_rep).
    const int bkv = (bh / Hq) * (Hq / n_rep) + (bh % Hq) / n_rep;
    const int n_kv = CAUSAL ? qt + 1 : n_tiles;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(Bar::QD_FULL), 1);
        for (int s = 0; s < C::NSK; ++s) {
            mbar_init(bar(Bar::K_FULL + s), 1);
            mbar_init(bar(Bar::K_EMPTY + s), 1);
        }
        for (int s = 0; s < C::NSV; ++s) {
            mbar_init(bar(Bar::V_FULL + s), 1);
            mbar_init(bar(Bar::V_EMPTY + s), 1);
        }
        mbar_init(bar(Bar::S_FULL), 1);
        mbar_init(bar(Bar::S_FULL + 1), 1);
        mbar_init(bar(Bar::DP_FULL), 1);
        mbar_init(bar(Bar::DP_EMPTY), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::DS_FULL), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::DS_FULL + 1), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::O_FULL), 1);
        mbar_init(bar(Bar::O_FREE), 1);
        mbar_init(bar(Bar::D_FULL), 1);
        mbar_init(bar(Bar::DQ_DONE), 1);
        mbar_init(bar(Bar::DONE), 2);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_do);
        if (fused) prefetch_tensormap(&tm_o);
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
    pdl_wait_then_release();

    if (warp == 0) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            // O first (fused first step): it is on the math warps' path to
            // their first dS.  It lands in K stage 2, free until K_2.
            const uint32_t s_o = s_k + 2 * C::TILE_BYTES;
            if (fused) {
                mbar_arrive_expect_tx(bar(Bar::O_FULL), C::TILE_BYTES);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_3d(s_o + kb * C::BOX_BYTES, &tm_o, bar(Bar::O_FULL), kb * 64,
                                qt * C::BM, bh);
            }
            mbar_arrive_expect_tx(bar(Bar::QD_FULL), 2 * C::TILE_BYTES);
            for (int kb = 0; kb < C::KB; ++kb) {
                tma_load_3d(s_q + kb * C::BOX_BYTES, &tm_q, bar(Bar::QD_FULL), kb * 64,
                            qt * C::BM, bh);
                tma_load_3d(s_do + kb * C::BOX_BYTES, &tm_do, bar(Bar::QD_FULL), kb * 64,
                            qt * C::BM, bh);
            }
            int issued = 0;
            for (; issued < n_kv; ++issued) {
                const int st = issued % C::NSK, use = issued / C::NSK;
                if (use > 0 && !mbar_wait(bar(Bar::K_EMPTY + st), (use - 1) & 1, wc)) break;
                if (fused && issued == 2 && !mbar_wait(bar(Bar::O_FREE), 0, wc)) break;
                mbar_arrive_expect_tx(bar(Bar::K_FULL + st), C::TILE_BYTES);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_3d(s_k + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_k,
                                bar(Bar::K_FULL + st), kb * 64, issued * C::BN, bkv);
            }
            if (fused) mbar_wait_drain(bar(Bar::O_FULL), 0, timeout_ns);
            mbar_wait_drain(bar(Bar::QD_FULL), 0, timeout_ns);
            for (int j = (issued > C::NSK ? issued - C::NSK : 0); j < issued; ++j)
                mbar_wait_drain(bar(Bar::K_FULL + j % C::NSK), (j / C::NSK) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == 11) {
        if (lane == 0) {
            int issued = 0;
            for (; issued < n_kv; ++issued) {
                const int st = issued % C::NSV, use = issued / C::NSV;
                if (use > 0 && !mbar_wait(bar(Bar::V_EMPTY + st), (use - 1) & 1, wc)) break;
                mbar_arrive_expect_tx(bar(Bar::V_FULL + st), C::TILE_BYTES);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_3d(s_v + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_v,
                                bar(Bar::V_FULL + st), kb * 64, issued * C::BN, bkv);
            }
            for (int j = (issued > C::NSV ? issued - C::NSV : 0); j < issued; ++j)
                mbar_wait_drain(bar(Bar::V_FULL + j % C::NSV), (j / C::NSV) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer A
        // Each issuer is a whole warp: every lane waits and computes the
        // operands, one elected lane issues the MMAs and commits.  Under a
        // causal mask issuer A is lane 0 alone instead: measured both ways,
        // the whole warp made dQ 5 % faster without the mask and 2-3 % slower
        // with it (the cause was not found).
        constexpr bool kWarpA = !CAUSAL;
        auto wait_a = [&](uint32_t b, uint32_t parity) {
            return kWarpA ? mbar_wait_warp(b, parity, wc) : mbar_wait(b, parity, wc);
        };
        auto lead_a = [&]() { return kWarpA ? elect_one() : true; };
        auto sync_a = [&]() {
            if (kWarpA) __syncwarp();
        };
        if (kWarpA || lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);  // S: both K-major
            constexpr uint32_t id_q = idesc_bf16(128, D, 0, 1);    // dQ: B MN-major
            const uint64_t d_q = smem_desc_sw128(s_q, 16, 1024);
            const uint64_t d_kk = smem_desc_sw128(s_k, 16, 1024);            // K, K-major
            const uint64_t d_kmn = smem_desc_sw128(s_k, C::BOX_BYTES, 1024);  // K, MN-major
            auto issue_s = [&](int j) -> bool {  // S_j = Q K_j^T into buffer j & 1
                const int st = j % C::NSK;
                if (!wait_a(bar(Bar::K_FULL + st), (j / C::NSK) & 1)) return false;
                tc_fence_after();
                const uint32_t d_tmem = tmem + ((j & 1) ? C::COL_S1 : C::COL_S0);
                const uint64_t d_b = desc_advance(d_kk, st * C::TILE_BYTES);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                    const uint64_t ad = desc_advance(d_q, koff);
                    const uint64_t bd = desc_advance(d_b, koff);
                    if (lead_a()) mma_ss(d_tmem, ad, bd, id_s, kk > 0);
                    sync_a();
                }
                if (lead_a()) tc_commit(bar(Bar::S_FULL + (j & 1)));
                sync_a();
                return true;
            };
            bool ok = wait_a(bar(Bar::QD_FULL), 0) && issue_s(0);
            if (ok && n_kv > 1) ok = issue_s(1);
            for (int j = 0; j < n_kv && ok; ++j) {
                const int st = j % C::NSK;
                ok = wait_a(bar(Bar::DS_FULL + (j & 1)), (j >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t s_cols = tmem + ((j & 1) ? C::COL_S1 : C::COL_S0);
                const uint64_t d_b = desc_advance(d_kmn, st * C::TILE_BYTES);
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {  // dQ += dS_j K_j
                    // dS halves: keys 0-63 at columns [0,32), 64-127 at [64,96).
                    const uint32_t scol = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
                    const uint64_t bd = desc_advance(d_b, kk * 2048);
                    if (lead_a())
                        mma_ts(tmem + C::COL_DQ, s_cols + scol, bd, id_q,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    sync_a();
                }
                if (lead_a()) tc_commit(bar(Bar::K_EMPTY + st));
                sync_a();
                if (j + 2 < n_kv) ok = issue_s(j + 2);
            }
            if (ok && lead_a()) tc_commit(bar(Bar::DQ_DONE));
            sync_a();
        }
        __syncwarp();
    } else if (warp == 10) {
        // ------------------------------------------------------------ MMA issuer B
        {
            constexpr uint32_t id_p = idesc_bf16(128, 128, 0, 0);  // dP: both K-major
            const uint64_t d_do = smem_desc_sw128(s_do, 16, 1024);
            const uint64_t d_vv = smem_desc_sw128(s_v, 16, 1024);
            auto issue_dp = [&](int j) -> bool {  // dP_j = dO V_j^T
                const int st = j % C::NSV;
                if (!mbar_wait_warp(bar(Bar::V_FULL + st), (j / C::NSV) & 1, wc)) return false;
                tc_fence_after();
                const uint64_t d_b = desc_advance(d_vv, st * C::TILE_BYTES);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                    const uint64_t ad = desc_advance(d_do, koff);
                    const uint64_t bd = desc_advance(d_b, koff);
                    if (elect_one()) mma_ss(tmem + C::COL_DP, ad, bd, id_p, kk > 0);
                    __syncwarp();
                }
                if (elect_one()) {
                    tc_commit(bar(Bar::V_EMPTY + st));
                    tc_commit(bar(Bar::DP_FULL));
                }
                __syncwarp();
                return true;
            };
            bool ok = mbar_wait_warp(bar(Bar::QD_FULL), 0, wc);
            if (ok && fused) {
                // The first backward step on the tensor core: dO O^T into the
                // dQ columns (free until the first dQ product), whose
                // diagonal is D_r = sum_c dO_rc O_rc.  Both operands K-major,
                // O in the K stage it arrived in.
                ok = mbar_wait_warp(bar(Bar::O_FULL), 0, wc);
                if (ok) {
                    tc_fence_after();
                    const uint64_t d_o = smem_desc_sw128(s_k + 2 * C::TILE_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                        const uint64_t ad = desc_advance(d_do, koff);
                        const uint64_t bd = desc_advance(d_o, koff);
                        if (elect_one()) mma_ss(tmem + C::COL_DQ, ad, bd, id_p, kk > 0);
                        __syncwarp();
                    }
                    if (elect_one()) {
                        tc_commit(bar(Bar::D_FULL));
                        tc_commit(bar(Bar::O_FREE));  // O has been read: K_2 may take its stage
                    }
                    __syncwarp();
                }
            }
            ok = ok && issue_dp(0);
            for (int j = 0; j + 1 < n_kv && ok; ++j)  // the math warps hold dP_j in registers
                ok = mbar_wait_warp(bar(Bar::DP_EMPTY), j & 1, wc) && issue_dp(j + 1);
        }
    } else {
        // ------------------------------------------------------------ P / dS
        const int wq = warp & 3;
        const int h = (warp - 2) >> 2;       // key half
        const int r = wq * 32 + lane;        // query row
        const int qglob = qt * C::BM + r;    // query index inside the head
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const long long voff = static_cast<long long>(bh) * n_pad + qt * C::BM + r;
        bool ok = true;
        float d_r, l2_r;  // D_r and LSE_r log2(e); 0 and +inf on padding rows
        if (fused) {
            // The first backward step, fused: D_r is the diagonal entry
            // (r, r) of dO O^T, which issuer B computes into the dQ columns;
            // lane r of this warp's quarter finds it at column r.
            const bool real = qglob < N;
            // LSE is issued first, so its latency runs under the waits.
            const float lse_r = real ? lse[static_cast<long long>(bh) * N + qglob] : 0.f;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::D_FULL), 0, wc));
            float dg = 0.f;
            if (ok) {
                tc_fence_after();
                uint32_t a[32];
                tmem_ld32(t_lane + C::COL_DQ + 32 * wq, a);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i == lane) dg = __uint_as_float(a[i]);
                tc_fence_before();
            }
            d_r = real ? dg : 0.f;
            l2_r = real ? lse_r * 1.4426950408889634f : INFINITY;
            if (h == 0) {
                delta[voff] = d_r;
                lse2[voff] = l2_r;
            }
        } else {
            d_r = delta[voff];
            l2_r = lse2[voff];
        }
        // P = 0 on padding rows (l2_r = +inf); log2(scale) folds scale into P.
        const float neg_l2 = log2f(scale) - l2_r;
        const float2 c2 = make_float2(scale_log2, scale_log2);
        const float2 neg_l2_2 = make_float2(neg_l2, neg_l2);
        const float2 neg_d2 = make_float2(-d_r, -d_r);  // dP - D as an addition of -D
        for (int j = 0; ok && j < n_kv; ++j) {
            const uint32_t t_s = t_lane + ((j & 1) ? C::COL_S1 : C::COL_S0) + 64 * h;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::S_FULL + (j & 1)), (j >> 1) & 1, wc) &&
                                             mbar_wait(bar(Bar::DP_FULL), j & 1, wc));
            if (!ok) break;
            tc_fence_after();
            const int key0 = j * C::BN + 64 * h;  // key index of entry 0
            const bool masked = (CAUSAL && j == qt) || key0 + 64 > N;
            // dP_j into registers first, so the next dP can be computed meanwhile.
            uint32_t dr[64];
            tmem_ld64(t_lane + C::COL_DP + 64 * h, dr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::DP_EMPTY));
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {  // two chunks of 32 keys
                uint32_t sr[32], w[16];
                tmem_ld32(t_s + 32 * ch, sr);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c = 2 * e;
                    const float2 x = fma2(make_float2(__uint_as_float(sr[c]),
                                                      __uint_as_float(sr[c + 1])),
                                          c2, neg_l2_2);
                    float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    if (masked) {
                        const int key = key0 + 32 * ch + c;
                        if ((CAUSAL && key > qglob) || key >= N) p.x = 0.f;
                        if ((CAUSAL && key + 1 > qglob) || key + 1 >= N) p.y = 0.f;
                    }
                    const float2 t = add2(make_float2(__uint_as_float(dr[32 * ch + c]),
                                                      __uint_as_float(dr[32 * ch + c + 1])),
                                          neg_d2);
                    const float2 ds = mul2(p, t);
                    w[e] = pack_bf16x2(ds.x, ds.y);
                }
                // Chunk ch's dS lands on S columns [16 ch, 16 ch + 16) of this
                // half, which chunk 0 has already read.
                tmem_st16(t_s + 16 * ch, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::DS_FULL + (j & 1)));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::DQ_DONE), 0, wc));
        if (ok) {
            // Every MMA has completed, so Q and dO (512 d bytes, the size of
            // the FP32 dQ tile) hold the staging boxes: this warp's 32 rows x
            // d/2 columns as d/64 boxes of 32 x 32, stored by TMA in whole
            // 128-byte rows.
            tc_fence_after();
            const uint32_t stg = s_q + static_cast<uint32_t>((warp - 2) * (D / 64) * 4096);
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch) {
                uint32_t a[32];
                tmem_ld32(t_lane + C::COL_DQ + (D / 2) * h + ch * 32, a);
                st_row_sw128_f32(stg + ch * 4096, lane, a, 1.f);
            }
            fence_async_smem();
            __syncwarp();
            const int row0 = qt * C::BM + wq * 32;
            if (lane == 0 && row0 < N) {
#pragma unroll
                for (int ch = 0; ch < D / 64; ++ch)
                    tma_store_3d(&tm_dq, stg + ch * 4096, (D / 2) * h + ch * 32, row0, bh);
                bulk_commit();
                bulk_wait_read_all();  // the boxes stay in place until read
            }
            __syncwarp();
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    // The commits come from the lane that issued each warp's MMAs.
    if (warp == 10 && elect_one()) tc_commit(bar(Bar::DONE));
    if (warp == 1) {
        if (CAUSAL ? lane == 0 : elect_one()) {
            tc_commit(bar(Bar::DONE));  // both issuers' MMAs have completed
            mbar_wait_drain(bar(Bar::DONE), 0, timeout_ns);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const DqArgs& a, cudaStream_t stream) {
    using C = DqCfg<D>;
    auto kern = bwd_dq_bf16_kernel<D, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.N + C::BM - 1) / C::BM;
    int group = 128 / n_tiles;
    if (group < 1) group = 1;
    dim3 grid(n_tiles, a.H, a.B);
    const bool fused = a.o != nullptr;
    e = launch_overlapped(kern, grid, dim3(C::THREADS), C::SMEM_BYTES, stream, *a.tm_q, *a.tm_k,
                          *a.tm_v, *a.tm_do, *a.tm_dq, fused ? *a.tm_o : *a.tm_q,
                          fused ? 1 : 0, a.lse,
                          a.delta, a.lse2, a.N, a.n_pad, a.B * a.H, a.H, a.H / a.Hkv, n_tiles,
                          group, a.scale, a.scale_log2, a.status, a.timeout_ns);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_bf16(const DqArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
    return a.causal ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
}

}  // namespace fa
