// bwd_dq_sm103.cu - attention backward, dQ kernel, BF16 in / FP32 out,
// tcgen05 + TMEM + TMA on sm_103a.
//
// Method.  dQ = scale dS K with dS = P o (dP - D), P = exp(scale Q K^T - LSE)
// recomputed from the saved LSE ("Flash Attention: Revolutionizing
// Transformer Efficiency", section "The Flash Attention algorithm", idea 2,
// recomputation) and dP = dO V^T.  A Q tile (128 rows of one (b, h)) is
// one work item: its CTA loops over the key tiles it sees (j <= i when
// causal), exactly like the forward's loop order ("FlashAttention scaling,
// multi-GPU training and weight quantization", section 1); the dQ tile
// accumulates in TMEM and is written once, so the result does not depend on
// the order in which CTAs run (no atomics; "FlashAttention-2" stresses a
// deterministic exact result).  The grid is persistent (one CTA per SM, at
// most one per item) and each CTA claims items from a counter, so a tile's
// loads and first products overlap the previous tile's last ones and its
// epilogue.
//
// Roles (384 threads, one CTA per SM):
//   warp 0      claimer and TMA producer: claims the next item and publishes
//               it in a small queue, then per tile Q_i and dO_i once the
//               previous tile's last S and dP products have read theirs,
//               (given O) the O tile into the next slot of a three-deep K
//               ring, K_j into the ring (K_j is read until the dQ MMA of tile
//               j), and at d = 128 the tile's staging slot.
//   warp 11     TMA producer: V_j into a two-deep ring (read only by dP_j).
//               The two rings free at different times, so each has its own
//               thread, and each thread its own warp: two lanes of one warp
//               that both spin on barriers share one instruction stream.
//   warps 1, 10 two MMA issuers.  Issuer A: S_0, S_1, then per key tile j:
//               dQ += dS_j K_j (A = dS_j in TMEM, after DS_FULL) and
//               S_j+2 = Q K_j+2^T over dS_j.  Issuer B: (given O)
//               D = diag(dO O^T) into the dQ columns once the math warps have
//               read the previous tile's dQ, dP_0, then dP_j+1 = dO V_j+1^T as
//               soon as the math warps hold dP_j in registers.  S is double
//               buffered and dP is released early, so both operands of tile
//               j+1 are ready when the math of tile j ends.
//   warps 2..9  thread (r, h) owns query row r (TMEM lane r) and key half h.
//               Given O and LSE, the backward's first step for their rows
//               comes first: D_r = sum_c dO_rc O_rc is the diagonal of dO O^T,
//               which issuer B computes on the tensor core into the dQ
//               columns; each thread reads its diagonal entry and writes D and
//               LSE2_r = LSE_r log2 e out for the dK/dV kernel.  Else they
//               read both.
//               Per key tile:
//               P' = exp2(S * scale*log2e - LSE2_r + log2 scale) = scale P,
//               dS' = P' o (dP - D_r) = scale dS, BF16, written over the first
//               32 of its own 64 S columns.  At the end: the dQ row half out
//               of TMEM, through a shared-memory box per warp, to global
//               memory (FP32) in whole 128-byte rows.
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
    static constexpr int BM = 128;  // query rows per Q tile
    static constexpr int BN = 128;  // keys per tile
    static constexpr int KB = D / 64;
    static constexpr int BOX_BYTES = 128 * 64 * 2;
    static constexpr int TILE_BYTES = KB * BOX_BYTES;
    static constexpr int NSK = 3;    // K ring depth (the O tile takes a slot too)
    static constexpr int NSV = 2;    // V ring depth
    static constexpr int QUEUE = 4;  // claimed-tile queue depth
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + TILE_BYTES;
    static constexpr int OFF_K = OFF_DO + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NSK * TILE_BYTES;
    // At d = 128 a tile's FP32 dQ passes through a K-ring slot of its own
    // (a slot position after the tile's last K tile) on its way to global
    // memory; at d = 64 through an area of its own (32 KB, room to spare).
    static constexpr bool STG_IN_K = (D == 128);
    static constexpr int OFF_STG = OFF_V + NSV * TILE_BYTES;
    static constexpr int STG_BYTES = STG_IN_K ? 0 : 8 * 4096;
    static constexpr int OFF_BAR = OFF_STG + STG_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int OFF_ITEMS = OFF_BAR + BAR_BYTES;
    static constexpr int LAYOUT_BYTES = OFF_ITEMS + QUEUE * 16;  // 4 ints per queued tile
    static constexpr int SMEM_BYTES =
        (LAYOUT_BYTES + 1024 <= kMaxDynSmem) ? LAYOUT_BYTES + 1024 : kMaxDynSmem;
    static_assert(LAYOUT_BYTES <= kMaxDynSmem, "dQ tiles do not fit in shared memory");
    // One 4 KB box (32 rows x 32 FP32 columns) per math warp.
    static_assert(!STG_IN_K || 8 * 4096 <= TILE_BYTES, "staging boxes fit a K slot");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_DP = 256, COL_DQ = 384;
    static constexpr int THREADS = 384;
    static constexpr int COMPUTE_WARPS = 8;
    // Arrivals on ITEM_EMPTY: both issuers, the V producer and 8 math warps
    // (the K producer writes the queue).
    static constexpr int ITEM_READERS = 11;
};

template <int NSK, int NSV, int QUEUE>
struct DqBars {
    static constexpr int QD_FULL = 0;
    // Q and dO are free for the next tile once both issuers' last products
    // that read them (the tile's last S and last dP) have run.
    static constexpr int QD_EMPTY = QD_FULL + 1;
    static constexpr int K_FULL = QD_EMPTY + 1;
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
    static constexpr int D_FULL = DS_FULL + 2;    // dO O^T in the dQ columns
    static constexpr int DQ_DONE = D_FULL + 1;
    static constexpr int DQ_FREE = DQ_DONE + 1;   // the math warps have read dQ
    // A staging slot is released by the math warps (one arrival each) once
    // they have read their boxes back; it completes one phase per tile.
    static constexpr int STG_FREE = DQ_FREE + 1;
    static constexpr int ITEM_FULL = STG_FREE + 1;  // QUEUE
    static constexpr int ITEM_EMPTY = ITEM_FULL + QUEUE;
    static constexpr int DONE = ITEM_EMPTY + QUEUE;
    static constexpr int COUNT = DONE + 1;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_o, int fused,
                       const float* __restrict__ lse, float* __restrict__ dq,
                       float* __restrict__ delta, float* __restrict__ lse2, int N, int n_pad, int BH,
                       int Hq, int n_rep, int n_tiles, int group,
                       float scale, float scale_log2, unsigned int* status,
                       unsigned long long timeout_ns, unsigned int* work) {
    using C = DqCfg<D>;
    using Bar = DqBars<C::NSK, C::NSV, C::QUEUE>;
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
    volatile int* items = reinterpret_cast<volatile int*>(smem + C::OFF_ITEMS);
    const int n_items = BH * n_tiles;

    // A work item is one Q tile of one (b, h): heavy Q tiles first (the last
    // Q tile sees the most keys under a causal mask), a few heads at a time
    // so that their K and V stay in L2.
    struct Tile {
        int qt, bh, bkv, n_kv;
    };
    auto tile_of = [&](int item) -> Tile {
        // Head groups in reverse: the forward before this kernel walks them
        // forwards, so the first Q tiles here find their Q, K, V and O in L2.
        const TileHead th = grouped_order(item, BH, n_tiles, group, true, true);
        Tile t;
        t.qt = th.tile;
        t.bh = th.head;
        // K/V head of query head bh: its group's head (b * Hkv + h / n_rep).
        t.bkv = (t.bh / Hq) * (Hq / n_rep) + (t.bh % Hq) / n_rep;
        t.n_kv = CAUSAL ? t.qt + 1 : n_tiles;
        return t;
    };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(Bar::QD_FULL), 1);
        mbar_init(bar(Bar::QD_EMPTY), 2);
        for (int s = 0; s < C::NSK; ++s) {
            mbar_init(bar(Bar::K_FULL + s), 1);
            mbar_init(bar(Bar::K_EMPTY + s), 1);
        }
        for (int s = 0; s < C::NSV; ++s) {
            mbar_init(bar(Bar::V_FULL + s), 1);
            mbar_init(bar(Bar::V_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(Bar::S_FULL + b), 1);
            mbar_init(bar(Bar::DS_FULL + b), C::COMPUTE_WARPS);
        }
        mbar_init(bar(Bar::DP_FULL), 1);
        mbar_init(bar(Bar::DP_EMPTY), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::D_FULL), 1);
        mbar_init(bar(Bar::DQ_DONE), 1);
        mbar_init(bar(Bar::DQ_FREE), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::STG_FREE), C::COMPUTE_WARPS);
        for (int i = 0; i < C::QUEUE; ++i) {
            mbar_init(bar(Bar::ITEM_FULL + i), 1);
            mbar_init(bar(Bar::ITEM_EMPTY + i), C::ITEM_READERS);
        }
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

    // Tile k of this CTA from the queue, as the claimer decoded it; qt = -1
    // at the end of the work or when a wait gave up.  The lane form is for a
    // single thread, the warp form for a whole warp (one arrival either way).
    auto read_item = [&](int slot) -> Tile {
        Tile t;
        t.qt = items[4 * slot];
        t.bh = items[4 * slot + 1];
        t.bkv = items[4 * slot + 2];
        t.n_kv = items[4 * slot + 3];
        return t;
    };
    auto take_item = [&](int k) -> Tile {
        const int slot = k % C::QUEUE;
        if (!mbar_wait(bar(Bar::ITEM_FULL + slot), (k / C::QUEUE) & 1, wc)) return Tile{-1, 0, 0, 0};
        const Tile t = read_item(slot);
        mbar_arrive(bar(Bar::ITEM_EMPTY + slot));
        return t;
    };
    auto take_item_warp = [&](int k) -> Tile {
        const int slot = k % C::QUEUE;
        if (!mbar_wait_warp(bar(Bar::ITEM_FULL + slot), (k / C::QUEUE) & 1, wc)) return Tile{-1, 0, 0, 0};
        const Tile t = read_item(slot);
        __syncwarp();
        if (elect_one()) mbar_arrive(bar(Bar::ITEM_EMPTY + slot));
        __syncwarp();
        return t;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ claimer + K producer
        if (lane == 0) {
            // Per tile: claim it and publish it, then Q and dO once the
            // previous tile's last S and dP products have read them, then
            // (given O) the O tile into the next K slot, the K tiles, and at
            // d = 128 the tile's staging slot.  The next tile is claimed once
            // this one's slots are all issued.  K slots run on one counter
            // across tiles, so a tile's loads start while the previous tile's
            // last products and epilogue still run.
            int ks = 0;            // K slots issued
            int qd_issued = 0;     // Q/dO loads issued
            bool ok = true, claimed_last = false;
            // Per physical slot: its loads so far (freed by K_EMPTY), and
            // whether its last use was a staging slot (freed by STG_FREE,
            // then the index of that staging use), else -1.
            int k_loads[C::NSK] = {};
            int k_stg[C::NSK];
            for (int i = 0; i < C::NSK; ++i) k_stg[i] = -1;
            int n_stg = 0;      // staging slots issued
            int stg_freed = 0;  // staging releases seen, in order
            // Waits until staging use m has been released.  Staging use m + 1
            // is marked only after release m has been seen, so STG_FREE never
            // runs more than one phase ahead of stg_freed.
            auto wait_stg = [&](int m) -> bool {
                for (; stg_freed <= m; ++stg_freed)
                    if (!mbar_wait(bar(Bar::STG_FREE), stg_freed & 1, wc)) return false;
                return true;
            };
            // Waits until physical slot st's last use is over.
            auto slot_free = [&](int st) -> bool {
                if (k_stg[st] >= 0) return wait_stg(k_stg[st]);
                if (k_loads[st] > 0) return mbar_wait(bar(Bar::K_EMPTY + st), (k_loads[st] - 1) & 1, wc);
                return true;
            };
            auto k_slot = [&](const CUtensorMap* map, int x_rows, int y_head) -> bool {
                const int st = ks % C::NSK;
                if (!slot_free(st)) return false;
                ++k_loads[st];
                k_stg[st] = -1;
                mbar_arrive_expect_tx(bar(Bar::K_FULL + st), C::TILE_BYTES);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_3d(s_k + st * C::TILE_BYTES + kb * C::BOX_BYTES, map,
                                bar(Bar::K_FULL + st), kb * 64, x_rows, y_head);
                ++ks;
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int slot = k % C::QUEUE;
                if (k >= C::QUEUE)
                    ok = mbar_wait(bar(Bar::ITEM_EMPTY + slot), ((k / C::QUEUE) - 1) & 1, wc);
                if (!ok) break;
                int item = static_cast<int>(blockIdx.x);
                if (k > 0) {
                    const unsigned int t = atomicAdd(work, 1u);
                    item = static_cast<int>(gridDim.x + t);
                    if (item >= n_items) {
                        claimed_last = true;
                        // Every CTA ends with exactly one failed claim, so the
                        // one that draws the last number is the last to claim:
                        // it puts the counter back to zero for the next launch.
                        if (t == static_cast<unsigned int>(n_items) - 1u) atomicExch(work, 0u);
                    }
                }
                // The tile is decoded once, here, off the other roles' paths.
                const Tile t = item < n_items ? tile_of(item) : Tile{-1, 0, 0, 0};
                items[4 * slot] = t.qt;
                items[4 * slot + 1] = t.bh;
                items[4 * slot + 2] = t.bkv;
                items[4 * slot + 3] = t.n_kv;
                mbar_arrive(bar(Bar::ITEM_FULL + slot));
                if (t.qt < 0) break;
                if (ok && k >= 1) ok = mbar_wait(bar(Bar::QD_EMPTY), (k - 1) & 1, wc);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(Bar::QD_FULL), 2 * C::TILE_BYTES);
                for (int kb = 0; kb < C::KB; ++kb) {
                    tma_load_3d(s_q + kb * C::BOX_BYTES, &tm_q, bar(Bar::QD_FULL), kb * 64,
                                t.qt * C::BM, t.bh);
                    tma_load_3d(s_do + kb * C::BOX_BYTES, &tm_do, bar(Bar::QD_FULL), kb * 64,
                                t.qt * C::BM, t.bh);
                }
                qd_issued = k + 1;
                if (fused) ok = k_slot(&tm_o, t.qt * C::BM, t.bh);
                for (int j = 0; ok && j < t.n_kv; ++j) ok = k_slot(&tm_k, j * C::BN, t.bkv);
                if (ok && C::STG_IN_K) {
                    // The tile's staging slot: nothing to load (its K_FULL
                    // phase completes at once, keeping every slot's phases
                    // in step with the positions), and the epilogue frees it.
                    const int st = ks % C::NSK;
                    ok = slot_free(st) && (n_stg == 0 || wait_stg(n_stg - 1));
                    if (ok) {
                        k_stg[st] = n_stg++;
                        mbar_arrive(bar(Bar::K_FULL + st));
                        ++ks;
                    }
                }
            }
            // After giving up, still draw numbers until one fails, so that
            // the counter is put back to zero as on the normal path.
            while (!claimed_last) {
                const unsigned int t = atomicAdd(work, 1u);
                if (gridDim.x + t >= static_cast<unsigned int>(n_items)) {
                    claimed_last = true;
                    if (t == static_cast<unsigned int>(n_items) - 1u) atomicExch(work, 0u);
                }
            }
            // Drain: no copy may still be landing when the CTA exits.
            if (qd_issued > 0) mbar_wait_drain(bar(Bar::QD_FULL), (qd_issued - 1) & 1, timeout_ns);
            for (int j = (ks > C::NSK ? ks - C::NSK : 0); j < ks; ++j)
                mbar_wait_drain(bar(Bar::K_FULL + j % C::NSK), (j / C::NSK) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == 11) {
        // ------------------------------------------------------------ V producer
        if (lane == 0) {
            int vs = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const Tile t = take_item(k);
                if (t.qt < 0) break;
                for (int j = 0; ok && j < t.n_kv; ++j, ++vs) {
                    const int st = vs % C::NSV, use = vs / C::NSV;
                    if (use > 0) ok = mbar_wait(bar(Bar::V_EMPTY + st), (use - 1) & 1, wc);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(Bar::V_FULL + st), C::TILE_BYTES);
                    for (int kb = 0; kb < C::KB; ++kb)
                        tma_load_3d(s_v + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_v,
                                    bar(Bar::V_FULL + st), kb * 64, j * C::BN, t.bkv);
                }
            }
            for (int j = (vs > C::NSV ? vs - C::NSV : 0); j < vs; ++j)
                mbar_wait_drain(bar(Bar::V_FULL + j % C::NSV), (j / C::NSV) & 1, timeout_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer A
        // Each issuer is a whole warp: every lane waits and computes the
        // operands, one elected lane issues the MMAs and commits.  (Under a
        // causal mask a lone-lane issuer A once measured faster; that was
        // while the mask test sat inside the exponential loop.  With the
        // mask in its own pass the whole warp is 2.5-5 % faster there too.)
        auto wait_a = [&](uint32_t b, uint32_t parity) { return mbar_wait_warp(b, parity, wc); };
        auto lead_a = [&]() { return elect_one(); };
        auto sync_a = [&]() { __syncwarp(); };
        {
            constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);  // S: both K-major
            constexpr uint32_t id_q = idesc_bf16(128, D, 0, 1);    // dQ: B MN-major
            const uint64_t d_q = smem_desc_sw128(s_q, 16, 1024);
            const uint64_t d_kk = smem_desc_sw128(s_k, 16, 1024);            // K, K-major
            const uint64_t d_kmn = smem_desc_sw128(s_k, C::BOX_BYTES, 1024);  // K, MN-major
            int ks = 0;  // K slots (O slots included), as the producer counts them
            int gj = 0;  // key tiles of earlier Q tiles: S buffers and dS barriers
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const Tile t = take_item_warp(k);
                if (t.qt < 0) break;
                if (fused) ++ks;  // the O slot, read by issuer B
                const int k0 = ks;
                ks += t.n_kv + (C::STG_IN_K ? 1 : 0);  // and the staging slot
                // S_j = Q K_j^T into buffer (gj + j) & 1.
                auto issue_s = [&](int j) -> bool {
                    const int slot = k0 + j, st = slot % C::NSK;
                    if (!wait_a(bar(Bar::K_FULL + st), (slot / C::NSK) & 1)) return false;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (((gj + j) & 1) ? C::COL_S1 : C::COL_S0);
                    const uint64_t d_b = desc_advance(d_kk, st * C::TILE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                        const uint64_t ad = desc_advance(d_q, koff);
                        const uint64_t bd = desc_advance(d_b, koff);
                        if (lead_a()) mma_ss(d_tmem, ad, bd, id_s, kk > 0);
                        sync_a();
                    }
                    if (lead_a()) tc_commit(bar(Bar::S_FULL + ((gj + j) & 1)));
                    sync_a();
                    return true;
                };
                // After the tile's last S this issuer has done with Q.  (The
                // branch stays outside the elected lane's code: a branch
                // among the issuing lane's instructions slowed the issue.)
                auto release_q = [&]() {
                    if (lead_a()) tc_commit(bar(Bar::QD_EMPTY));
                    sync_a();
                };
                ok = wait_a(bar(Bar::QD_FULL), k & 1) && issue_s(0);
                if (ok && t.n_kv > 1) ok = issue_s(1);
                if (ok && t.n_kv <= 2) release_q();
                for (int j = 0; j < t.n_kv && ok; ++j) {
                    const int g = gj + j;
                    const int slot = k0 + j, st = slot % C::NSK;
                    ok = wait_a(bar(Bar::DS_FULL + (g & 1)), (g >> 1) & 1);
                    // The tile's first dQ product overwrites the accumulator:
                    // the math warps must have read the previous tile's out.
                    if (ok && j == 0 && k >= 1) ok = wait_a(bar(Bar::DQ_FREE), (k - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t s_cols = tmem + ((g & 1) ? C::COL_S1 : C::COL_S0);
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
                    if (j + 2 < t.n_kv) {
                        ok = issue_s(j + 2);
                        if (ok && j + 3 == t.n_kv) release_q();
                    }
                }
                if (ok && lead_a()) tc_commit(bar(Bar::DQ_DONE));
                sync_a();
                gj += t.n_kv;
            }
        }
        __syncwarp();
    } else if (warp == 10) {
        // ------------------------------------------------------------ MMA issuer B
        constexpr uint32_t id_p = idesc_bf16(128, 128, 0, 0);  // dP, D: both K-major
        const uint64_t d_do = smem_desc_sw128(s_do, 16, 1024);
        const uint64_t d_vv = smem_desc_sw128(s_v, 16, 1024);
        int ks = 0, vs = 0, gj = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const Tile t = take_item_warp(k);
            if (t.qt < 0) break;
            const int o_slot = ks;
            if (fused) ++ks;
            ks += t.n_kv + (C::STG_IN_K ? 1 : 0);
            const int v0 = vs;
            vs += t.n_kv;
            auto issue_dp = [&](int j) -> bool {  // dP_j = dO V_j^T
                const int slot = v0 + j, st = slot % C::NSV;
                if (!mbar_wait_warp(bar(Bar::V_FULL + st), (slot / C::NSV) & 1, wc)) return false;
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
            ok = mbar_wait_warp(bar(Bar::QD_FULL), k & 1, wc);
            if (ok && fused) {
                // The first backward step on the tensor core: dO O^T into the
                // dQ columns, whose diagonal is D_r = sum_c dO_rc O_rc.  Both
                // operands K-major, O in the K slot it arrived in.  The
                // columns are free once the math warps have read the previous
                // tile's dQ; the tile's first dQ product follows the math
                // warps' first dS, so they have read D by then.
                const int st = o_slot % C::NSK;
                if (k >= 1) ok = mbar_wait_warp(bar(Bar::DQ_FREE), (k - 1) & 1, wc);
                ok = ok && mbar_wait_warp(bar(Bar::K_FULL + st), (o_slot / C::NSK) & 1, wc);
                if (ok) {
                    tc_fence_after();
                    const uint64_t d_o = smem_desc_sw128(s_k + st * C::TILE_BYTES, 16, 1024);
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
                        tc_commit(bar(Bar::K_EMPTY + st));  // O has been read
                    }
                    __syncwarp();
                }
            }
            // The dP columns are free once the math warps hold the previous
            // tile's last dP in registers.
            if (ok && gj > 0) ok = mbar_wait_warp(bar(Bar::DP_EMPTY), (gj - 1) & 1, wc);
            ok = ok && issue_dp(0);
            for (int j = 0; j + 1 < t.n_kv && ok; ++j)  // the math warps hold dP_j in registers
                ok = mbar_wait_warp(bar(Bar::DP_EMPTY), (gj + j) & 1, wc) && issue_dp(j + 1);
            // After the tile's last dP this issuer has done with dO.
            if (ok) {
                if (elect_one()) tc_commit(bar(Bar::QD_EMPTY));
                __syncwarp();
            }
            gj += t.n_kv;
        }
    } else {
        // ------------------------------------------------------------ P / dS, epilogue
        const int wq = warp & 3;
        const int h = (warp - 2) >> 2;       // key half
        const int r = wq * 32 + lane;        // query row
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        int gj = 0;  // key tiles of earlier Q tiles
        int ks = 0;  // K slots, as the producer counts them (for the staging slot)
        bool ok = true;
        const float log2_scale = log2f(scale);
        // A tile's per-row inputs (LSE given O, else D and LSE2) are loaded
        // as soon as the tile is known: the next tile's while this one's
        // epilogue runs.
        struct RowIn {
            float a, b;
        };
        auto row_in = [&](const Tile& u) -> RowIn {
            RowIn v{0.f, 0.f};
            if (u.qt < 0) return v;
            const int qg = u.qt * C::BM + r;
            if (fused) {
                if (qg < N) v.a = lse[static_cast<long long>(u.bh) * N + qg];
            } else {
                const long long off = static_cast<long long>(u.bh) * n_pad + qg;
                v.a = delta[off];
                v.b = lse2[off];
            }
            return v;
        };
        Tile t = take_item_warp(0);
        RowIn in = row_in(t);
        for (int k = 0; ok && t.qt >= 0; ++k) {
            const int qt = t.qt, bh = t.bh;
            const int stg_pos = ks + (fused ? 1 : 0) + t.n_kv;  // this tile's staging slot
            ks = stg_pos + (C::STG_IN_K ? 1 : 0);
            const int qglob = qt * C::BM + r;    // query index inside the head
            const long long voff = static_cast<long long>(bh) * n_pad + qt * C::BM + r;
            float d_r, l2_r;  // D_r and LSE_r log2(e); 0 and +inf on padding rows
            if (fused) {
                // The first backward step, fused: D_r is the diagonal entry
                // (r, r) of dO O^T, which issuer B computes into the dQ
                // columns; lane r of this warp's quarter finds it at column r.
                const bool real = qglob < N;
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::D_FULL), k & 1, wc));
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
                __syncwarp();
                d_r = real ? dg : 0.f;
                l2_r = real ? in.a * 1.4426950408889634f : INFINITY;
                if (h == 0) {
                    delta[voff] = d_r;
                    lse2[voff] = l2_r;
                }
            } else {
                d_r = in.a;
                l2_r = in.b;
            }
            // P = 0 on padding rows (l2_r = +inf); log2(scale) folds scale into P.
            const float neg_l2 = log2_scale - l2_r;
            const float2 c2 = make_float2(scale_log2, scale_log2);
            const float2 neg_l2_2 = make_float2(neg_l2, neg_l2);
            const float2 neg_d2 = make_float2(-d_r, -d_r);  // dP - D as an addition of -D
            for (int j = 0; ok && j < t.n_kv; ++j) {
                const int g = gj + j;
                const uint32_t t_s = t_lane + ((g & 1) ? C::COL_S1 : C::COL_S0) + 64 * h;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(bar(Bar::S_FULL + (g & 1)), (g >> 1) & 1, wc) &&
                                    mbar_wait(bar(Bar::DP_FULL), g & 1, wc));
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
                    float p[32];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float2 x = fma2(make_float2(__uint_as_float(sr[c]),
                                                          __uint_as_float(sr[c + 1])),
                                              c2, neg_l2_2);
                        p[c] = ex2_approx(x.x);
                        p[c + 1] = ex2_approx(x.y);
                    }
                    // The mask in a pass of its own behind one branch: laid
                    // into the loop above, it is paid on every key tile.
                    if (masked) {
                        // Keys past the row (causal) or past N: entry c is
                        // kept while c < lim.
                        const int lim = (CAUSAL ? min(qglob + 1, N) : N) - (key0 + 32 * ch);
#pragma unroll
                        for (int c = 0; c < 32; ++c) p[c] = c < lim ? p[c] : 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c = 2 * e;
                        const float2 tt = add2(make_float2(__uint_as_float(dr[32 * ch + c]),
                                                           __uint_as_float(dr[32 * ch + c + 1])),
                                               neg_d2);
                        const float2 ds = mul2(make_float2(p[c], p[c + 1]), tt);
                        w[e] = pack_bf16x2(ds.x, ds.y);
                    }
                    // Chunk ch's dS lands on S columns [16 ch, 16 ch + 16) of this
                    // half, which chunk 0 has already read.
                    tmem_st16(t_s + 16 * ch, w);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Bar::DS_FULL + (g & 1)));
            }
            gj += t.n_kv;
            // The next tile now, so that its row inputs load under this epilogue.
            const Tile tn = ok ? take_item_warp(k + 1) : Tile{-1, 0, 0, 0};
            in = row_in(tn);
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::DQ_DONE), k & 1, wc));
            if (!ok) break;
            tc_fence_after();
            const int row0 = qt * C::BM + wq * 32;
            // dQ out of TMEM first (the columns are released at once), then
            // to global memory through one 4 KB box per warp (32 rows x 32
            // FP32 columns, d/64 rounds): each lane writes its row into the
            // box, then each store instruction of the warp moves four whole
            // 128-byte rows, eight lanes to a row.  At d = 128 the boxes lie
            // in the tile's own K slot, released once every warp has read
            // its box back.
            uint32_t a[D / 64][32];
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch)
                tmem_ld32(t_lane + C::COL_DQ + (D / 2) * h + ch * 32, a[ch]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::DQ_FREE));
            uint32_t box = s_base + C::OFF_STG + static_cast<uint32_t>((warp - 2) * 4096);
            if constexpr (C::STG_IN_K) {
                // The producer marks the slot as this tile's once its last
                // use is over; waiting for that mark also keeps this tile's
                // release (STG_FREE) behind the producer's wait for the
                // previous one.
                const int st = stg_pos % C::NSK;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(bar(Bar::K_FULL + st), (stg_pos / C::NSK) & 1, wc));
                if (!ok) break;
                box = s_k + st * C::TILE_BYTES + static_cast<uint32_t>((warp - 2) * 4096);
            }
            float* dq_rows = dq + (static_cast<long long>(bh) * N + row0) * D + (D / 2) * h;
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch) {
                st_row_sw128_f32(box, lane, a[ch], 1.f);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = 4 * i + (lane >> 3), c = lane & 7;
                    const float4 v = ld_shared_f4(box + rr * 128 + ((c ^ (rr & 7)) << 4));
                    if (row0 + rr < N)
                        *reinterpret_cast<float4*>(dq_rows + static_cast<long long>(rr) * D +
                                                   ch * 32 + 4 * c) = v;
                }
                __syncwarp();
            }
            if constexpr (C::STG_IN_K) {
                // The slot's next use is a TMA load over these generic writes.
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Bar::STG_FREE));
            }
            t = tn;
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    // The commits come from the lane that issued each warp's MMAs.
    if (warp == 10 && elect_one()) tc_commit(bar(Bar::DONE));
    if (warp == 1) {
        if (elect_one()) {
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
    const int group = claim_group(n_tiles, CAUSAL);
    // Persistent: one CTA per SM (at most one per Q tile) claims Q tiles.
    const long long n_items = static_cast<long long>(a.B) * a.H * n_tiles;
    const int grid = static_cast<int>(n_items < a.num_sms ? n_items : a.num_sms);
    const bool fused = a.o != nullptr;
    e = launch_overlapped(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, *a.tm_q,
                          *a.tm_k, *a.tm_v, *a.tm_do, fused ? *a.tm_o : *a.tm_q,
                          fused ? 1 : 0, a.lse, a.dq,
                          a.delta, a.lse2, a.N, a.n_pad, a.B * a.H, a.H, a.H / a.Hkv, n_tiles,
                          group, a.scale, a.scale_log2, a.status, a.timeout_ns, a.work);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_bf16(const DqArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
    return a.causal ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
}

}  // namespace fa
