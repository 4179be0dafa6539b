// fwd_bf16_sm103.cu - exact attention forward, BF16 in / FP32 accumulate,
// tcgen05 + TMEM + TMA on sm_103a.
//
// Method.  The online softmax of "LLM part 06: FlashAttention - GPU SRAM,
// tiling and online softmax" (section 2): each query row keeps a running max m
// and running sum l while key blocks stream past, and the output accumulator
// is rescaled by exp(m_old - m_new) whenever the max moves.  Loop order and
// parallelism follow "FlashAttention scaling, multi-GPU training and weight
// quantization" (section 1): one 128-row Q tile of one (batch, head) at a
// time, the K/V tiles in the inner loop, TMA copies issued by a producer warp,
// and the division by l deferred to the end ("FlashAttention-2", technical
// architecture, improvement 1).
//
// GB300 mapping: a persistent kernel, one CTA per SM (384 threads), that
// claims Q tiles from a per-launch counter (heavy tiles first, a few heads at
// a time so that their K/V tiles stay in L2).  Tiles run back to back: the
// next tile's Q is loaded and its first scores computed while the current
// one finishes, and its O store drains while the next one runs.
//   warp 0      loads K_j and V_j into NS-deep rings (128-byte swizzle,
//               64-column boxes), K one key tile ahead of V.
//   warp 3      claims tiles and loads each Q tile into one of two
//               shared-memory buffers.  It has a warp of its own: two lanes
//               of one warp that both spin on barriers share one instruction
//               stream, and the loads of one would wait on the other's spin.
//   warps 1, 2  two MMA issuers (whole warps; one elected lane issues).  A:
//               S_j = Q K_j^T (both operands in shared memory) into one of
//               three TMEM score buffers, once P V has read the probabilities
//               of S_{j-3} out of it.  B: O += P_j V_j (P from TMEM) as soon as
//               the softmax warps release P_j.  Three score buffers let S_{j+1}
//               run while P V_{j-1} and the softmax of tile j are in flight.
//   warps 4-11  softmax: thread (r, h) owns query row r (TMEM lane r) and
//               keys [64h, 64h+64) of every tile (warps 4-7: h = 0, 8-11:
//               h = 1), so two warps share each SM sub-partition's rows and
//               hide each other's latency.  Per tile: load its 64 scores, mask,
//               swap the partial row max with the partner warp through shared
//               memory, update m and its half of l, write P as BF16 over the
//               first half of its own score columns, and rescale its d/2
//               columns of the O accumulator (after PV_{j-1} has run) only when
//               the max grew by more than 2^8 (the final O / l and LSE use the
//               same stale max, so the result is unchanged).  After a Q tile's
//               last key tile the next tile is taken, so that its first score
//               MMAs run during this tile's epilogue: the two halves of l are
//               summed, O / l goes to BF16 into the tile's Q buffer (its score
//               MMAs are done) and out by TMA store; LSE = ln 2 * (m + log2 l).
// Warpgroup 0 (warps 0-3) hands registers to the softmax warpgroups, which
// hold a row half of scores, probabilities and O in flight.
//
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+d), S2 [256+d,
// 384+d); tile j's P as BF16 pairs at [0,32) and [64,96) of its score
// buffer.  All waits are bounded (see sm103_primitives.cuh); a CTA that gives
// up tells the others through its abort flag and every role leaves at its
// next wait.
#include "fa_internal.h"
#include "sm103_fp8.cuh"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kMaxDynSmem = 232448;  // 227 KB opt-in limit per block
constexpr uint32_t kRegsLight = 64;     // warps 0-3 after the split
constexpr uint32_t kRegsSoftmax = 216;  // warps 4-11 after the split
static_assert(128 * (kRegsLight + 2 * kRegsSoftmax) <= 384 * 168, "register split");
constexpr int kStoreThread = 128;       // softmax thread that issues the O stores

template <int D, bool FP8 = false>
struct FwdCfg {
    static constexpr int BM = 128;                    // query rows per tile
    static constexpr int BN = 128;                    // keys per K/V tile
    static constexpr int KB = D / 64;                 // 64-column (128-byte) boxes per row
    static constexpr int BOX_BYTES = 128 * 64 * 2;    // one 128 x 64 bf16 box
    static constexpr int TILE_BYTES = KB * BOX_BYTES; // one 128 x D bf16 tile
    // FP8: Q and K tiles are 128 x D E4M3 codes, one box of D-byte rows
    // (128-byte swizzle at D = 128, 64-byte swizzle at D = 64).
    static constexpr int QK_BYTES = FP8 ? 128 * D : TILE_BYTES;
    static constexpr int NS = (D == 128) ? 2 : 4;     // K/V ring depth
    static constexpr int QUEUE = 4;                   // claimed-tile queue depth
    // Two Q buffers of a BF16 tile each: the O tile is staged over them.
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NS * QK_BYTES;
    static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int OFF_XCH = OFF_BAR + BAR_BYTES;  // row maxima and sums of the halves
    static constexpr int XCH_BYTES = 6 * 128 * 4;
    static constexpr int OFF_ITEMS = OFF_XCH + XCH_BYTES;
    static constexpr int LAYOUT_BYTES = OFF_ITEMS + QUEUE * 4;
    static constexpr int SMEM_BYTES = LAYOUT_BYTES + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= kMaxDynSmem, "forward tiles do not fit in shared memory");
    static constexpr uint32_t TMEM_COLS = 512;
    // Three FP32 score buffers (S0, S1 around the O accumulator, S2 after
    // it); the BF16 P of each tile is written over the first half of its own
    // scores.  Q stays in shared memory.
    static constexpr int NSB = 3;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256, COL_S2 = COL_O + D;
    static_assert(COL_S2 + BN <= TMEM_COLS, "TMEM columns");
    __device__ static constexpr uint32_t col_s(int b) {
        return b == 0 ? COL_S0 : (b == 1 ? COL_S1 : COL_S2);
    }
    static constexpr int THREADS = 384;
    // Arrivals on ITEM_EMPTY: the K/V producer, both issuers, 8 softmax warps.
    static constexpr int ITEM_READERS = 11;
};

// Barrier slots (8 bytes each) inside the barrier area.
template <int NS, int QUEUE>
struct FwdBars {
    static constexpr int Q_FULL = 0;               // 2
    static constexpr int Q_EMPTY = Q_FULL + 2;     // 2
    static constexpr int K_FULL = Q_EMPTY + 2;
    static constexpr int V_FULL = K_FULL + NS;
    static constexpr int K_EMPTY = V_FULL + NS;
    static constexpr int V_EMPTY = K_EMPTY + NS;
    // One S_FULL / S_EMPTY / P_FULL triple per score buffer.
    static constexpr int S_FULL = V_EMPTY + NS;    // 3
    static constexpr int S_EMPTY = S_FULL + 3;     // 3
    static constexpr int P_FULL = S_EMPTY + 3;     // 3
    static constexpr int ITEM_FULL = P_FULL + 3;   // QUEUE
    static constexpr int ITEM_EMPTY = ITEM_FULL + QUEUE;
    static constexpr int CLAIM_OK = ITEM_EMPTY + QUEUE;
    static constexpr int DONE = CLAIM_OK + 1;
    static constexpr int COUNT = DONE + 1;
};

template <int D, bool CAUSAL, bool SPLIT, bool FP8>
__global__ void __launch_bounds__(384, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, float* __restrict__ lse, int N,
                    int BH, int Hq, int n_rep, int n_tiles, int group, float scale_log2,
                    unsigned int* status, unsigned long long timeout_ns, unsigned int* work,
                    int Nk, int n_splits, int chunk_tiles, float* __restrict__ o_part,
                    float* __restrict__ lse_part, const float* __restrict__ q_scale,
                    const float* __restrict__ k_scale) {
    using C = FwdCfg<D, FP8>;
    static_assert(!(FP8 && SPLIT), "the FP8 forward has no split mode");
    using Bar = FwdBars<C::NS, C::QUEUE>;
    static_assert(8 * Bar::COUNT + 8 <= C::BAR_BYTES, "barrier area");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    if (smem + C::LAYOUT_BYTES > smem_raw + C::SMEM_BYTES) {
        if (threadIdx.x == 0) atomicOr(status, kStatusSmemLayout);
        return;
    }
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + C::OFF_Q;
    const uint32_t s_k = s_base + C::OFF_K;
    const uint32_t s_v = s_base + C::OFF_V;
    const uint32_t s_bar = s_base + C::OFF_BAR;
    auto bar = [&](int slot) -> uint32_t { return s_bar + 8u * static_cast<uint32_t>(slot); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * Bar::COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* items = reinterpret_cast<volatile int*>(smem + C::OFF_ITEMS);
    // A work item is one Q tile of one head; with SPLIT, one Q tile of one
    // head against one chunk of key tiles (the key chunk varies fastest).
    const int n_items = BH * n_tiles * n_splits;
    const int n_kv_tiles = (Nk + C::BN - 1) / C::BN;
    struct Work {
        int qt, bh, s;  // Q tile, query head (b * Hq + h), key chunk
        int j0, j1;     // key tiles [j0, j1)
    };
    auto work_of = [&](int item) -> Work {
        Work w;
        w.s = SPLIT ? item % n_splits : 0;
        const TileHead th = grouped_order(SPLIT ? item / n_splits : item, BH, n_tiles, group, true);
        w.qt = th.tile;
        w.bh = th.head;
        if (SPLIT) {
            w.j0 = w.s * chunk_tiles;
            w.j1 = min(w.j0 + chunk_tiles, n_kv_tiles);
        } else {
            w.j0 = 0;
            w.j1 = CAUSAL ? th.tile + 1 : n_kv_tiles;
        }
        return w;
    };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(Bar::Q_FULL + b), 1);
            mbar_init(bar(Bar::Q_EMPTY + b), 1);
        }
        for (int b = 0; b < C::NSB; ++b) {
            mbar_init(bar(Bar::S_FULL + b), 1);
            mbar_init(bar(Bar::S_EMPTY + b), 1);  // P V of the buffer's P has run
            mbar_init(bar(Bar::P_FULL + b), 8);   // one arrival per softmax warp
        }
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(Bar::K_FULL + s), 1);
            mbar_init(bar(Bar::V_FULL + s), 1);
            mbar_init(bar(Bar::K_EMPTY + s), 1);
            mbar_init(bar(Bar::V_EMPTY + s), 1);
        }
        for (int i = 0; i < C::QUEUE; ++i) {
            mbar_init(bar(Bar::ITEM_FULL + i), 1);
            mbar_init(bar(Bar::ITEM_EMPTY + i), C::ITEM_READERS);
        }
        mbar_init(bar(Bar::CLAIM_OK), 1);
        mbar_init(bar(Bar::DONE), 2);  // one commit per issuer
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_o);
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

    // Tile k of this CTA from the queue (single-thread roles).  Returns -1 at
    // the end of the work or when a wait gave up.
    auto take_item = [&](int k) -> int {
        const int slot = k % C::QUEUE;
        if (!mbar_wait(bar(Bar::ITEM_FULL + slot), (k / C::QUEUE) & 1, wc)) return -1;
        const int item = items[slot];
        mbar_arrive(bar(Bar::ITEM_EMPTY + slot));
        return item;
    };
    // The same for a whole warp (the MMA issuers): one arrival per warp.
    auto take_item_warp = [&](int k) -> int {
        const int slot = k % C::QUEUE;
        if (!mbar_wait_warp(bar(Bar::ITEM_FULL + slot), (k / C::QUEUE) & 1, wc)) return -1;
        const int item = __shfl_sync(0xffffffffu, items[slot], 0);
        if (elect_one()) mbar_arrive(bar(Bar::ITEM_EMPTY + slot));
        __syncwarp();
        return item;
    };

    // Warpgroup 0 (warps 0-3: one thread each of real work) gives registers
    // to the softmax warpgroups 1 and 2:
    // 128 x (kRegsLight + 2 kRegsSoftmax) <= 384 x 168 at launch.
    if (warp < 4) {
        regs_decrease<kRegsLight>();
        if (warp == 3) {
            if (lane == 0) {
                // ------------------------------------------------ scheduler + Q loads
                // Tile k+1 is claimed once the K loads of tile k have all been
                // issued (a few key tiles before its end: early enough to hide the
                // Q load, late enough that the CTAs that finish first get the
                // remaining work), its Q buffer is free (the store of tile k-1 has
                // read it) and its queue slot has been read.
                int q_issued = 0;
                bool ok = true, claimed_last = false;
                for (int k = 0; ok; ++k) {
                    const int qb = k & 1;
                    const int slot = k % C::QUEUE;
                    if (k >= 1) ok = mbar_wait(bar(Bar::CLAIM_OK), (k - 1) & 1, wc);
                    if (ok && k >= 2) ok = mbar_wait(bar(Bar::Q_EMPTY + qb), ((k - 2) >> 1) & 1, wc);
                    if (ok && k >= C::QUEUE)
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
                    if (item >= n_items) item = -1;
                    items[slot] = item;
                    mbar_arrive(bar(Bar::ITEM_FULL + slot));
                    if (item < 0) break;
                    const Work w = work_of(item);
                    mbar_arrive_expect_tx(bar(Bar::Q_FULL + qb), C::QK_BYTES);
                    if constexpr (FP8) {
                        tma_load_3d(s_q + qb * C::TILE_BYTES, &tm_q, bar(Bar::Q_FULL + qb), 0,
                                    w.qt * C::BM, w.bh);
                    } else {
                        for (int kb = 0; kb < C::KB; ++kb)
                            tma_load_3d(s_q + qb * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_q,
                                        bar(Bar::Q_FULL + qb), kb * 64, w.qt * C::BM, w.bh);
                    }
                    q_issued = k + 1;
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
                for (int k = (q_issued > 2 ? q_issued - 2 : 0); k < q_issued; ++k)
                    mbar_wait_drain(bar(Bar::Q_FULL + (k & 1)), (k >> 1) & 1, timeout_ns);
            }
            __syncwarp();
        } else if (warp == 0) {
            if (lane == 0) {
                // ------------------------------------------------ K/V producer
                // K runs one key tile ahead of V over the stream of key tiles
                // of consecutive Q tiles: the next score MMAs need K_{g+1}
                // while P V_g still waits for V_g, and a K stage frees (after
                // its S) earlier than a V stage (after its P V).
                int k_issued = 0, v_issued = 0;
                bool ok = true;
                auto head_of = [&](int bh) { return (bh / Hq) * (Hq / n_rep) + (bh % Hq) / n_rep; };
                auto issue_k = [&](int j, int bkv) -> bool {
                    const int g = k_issued, st = g % C::NS, use = g / C::NS;
                    if (use > 0 && !mbar_wait(bar(Bar::K_EMPTY + st), (use - 1) & 1, wc)) return false;
                    mbar_arrive_expect_tx(bar(Bar::K_FULL + st), C::QK_BYTES);
                    if constexpr (FP8) {
                        tma_load_3d(s_k + st * C::QK_BYTES, &tm_k, bar(Bar::K_FULL + st), 0,
                                    j * C::BN, bkv);
                    } else {
                        for (int kb = 0; kb < C::KB; ++kb)
                            tma_load_3d(s_k + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_k,
                                        bar(Bar::K_FULL + st), kb * 64, j * C::BN, bkv);
                    }
                    k_issued = g + 1;
                    return true;
                };
                auto issue_v = [&](int j, int bkv) -> bool {
                    const int g = v_issued, st = g % C::NS, use = g / C::NS;
                    if (use > 0 && !mbar_wait(bar(Bar::V_EMPTY + st), (use - 1) & 1, wc)) return false;
                    mbar_arrive_expect_tx(bar(Bar::V_FULL + st), C::TILE_BYTES);
                    for (int kb = 0; kb < C::KB; ++kb)
                        tma_load_3d(s_v + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_v,
                                    bar(Bar::V_FULL + st), kb * 64, j * C::BN, bkv);
                    v_issued = g + 1;
                    return true;
                };
                // The K cursor: Q tile ck, key tile cj of it, K/V head cbkv.
                int ck = 0, cj = 0, cbkv = 0;
                Work cw{};
                // Moves the cursor to the next key tile, taking Q tiles from
                // the queue as it leaves one (and letting the next be claimed:
                // every K load of the tile left behind has been issued); false
                // at the end of the work.
                auto advance = [&]() -> bool {
                    ++cj;
                    while (cj >= cw.j1) {
                        mbar_arrive(bar(Bar::CLAIM_OK));
                        const int nitem = take_item(ck + 1);
                        if (nitem < 0) return false;
                        ++ck;
                        cw = work_of(nitem);
                        cj = cw.j0;
                        cbkv = head_of(cw.bh);
                    }
                    return true;
                };
                const int item0 = take_item(0);
                bool more = false;
                if (item0 >= 0) {
                    cw = work_of(item0);
                    cj = cw.j0 - 1;
                    cbkv = head_of(cw.bh);
                    more = advance();
                }
                if (more) ok = issue_k(cj, cbkv);
                while (more && ok) {
                    const int vj = cj, vbkv = cbkv;
                    more = advance();
                    if (more) ok = issue_k(cj, cbkv);
                    ok = ok && issue_v(vj, vbkv);
                }
                for (int t = (k_issued > C::NS ? k_issued - C::NS : 0); t < k_issued; ++t)
                    mbar_wait_drain(bar(Bar::K_FULL + t % C::NS), (t / C::NS) & 1, timeout_ns);
                for (int t = (v_issued > C::NS ? v_issued - C::NS : 0); t < v_issued; ++t)
                    mbar_wait_drain(bar(Bar::V_FULL + t % C::NS), (t / C::NS) & 1, timeout_ns);
            }
            __syncwarp();
        } else {  // warps 1, 2
            // ------------------------------------------------------------ MMA issuers
            // Each issuer is a whole warp: every lane waits and computes the
            // operands, one elected lane issues the MMAs and commits.
            constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);  // B = K, K-major
            constexpr uint32_t id_pv = idesc_bf16(128, D, 0, 1);   // B = V, MN-major
            int g = 0;  // tile counter across this CTA's Q tiles
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int item = take_item_warp(k);
                if (item < 0) break;
                const Work w = work_of(item);
                if (warp == 2) {
                    // Issuer B: O += P_j V_j as soon as the softmax warps release P_j.
                    for (int j = w.j0; j < w.j1 && ok; ++j, ++g) {
                        const int st = g % C::NS;
                        const int b = g % C::NSB;
                        ok = mbar_wait_warp(bar(Bar::P_FULL + b), (g / C::NSB) & 1, wc) &&
                             mbar_wait_warp(bar(Bar::V_FULL + st), (g / C::NS) & 1, wc);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t v_tile = s_v + st * C::TILE_BYTES;
                        // P_j (BF16) over its own scores: keys [64h, 64h+64) at
                        // columns [64h, 64h+32) of S buffer b.
                        const uint32_t p_cols = tmem + C::col_s(b);
#pragma unroll
                        for (int kk = 0; kk < C::BN / 16; ++kk) {
                            // V as an MN-major B operand: 16 keys = 2 atoms of 8 rows.
                            const uint64_t bd =
                                smem_desc_sw128(v_tile + kk * 2048, C::BOX_BYTES, 1024);
                            if (elect_one())
                                mma_ts(tmem + C::COL_O, p_cols + (kk >> 2) * 64 + (kk & 3) * 8, bd,
                                       id_pv, (j > w.j0 || kk > 0));
                            __syncwarp();
                        }
                        if (elect_one()) {
                            tc_commit(bar(Bar::V_EMPTY + st));
                            tc_commit(bar(Bar::S_EMPTY + b));  // P_j read: S buffer b is free
                        }
                        __syncwarp();
                    }
                } else {
                    // Issuer A: S_j = Q K_j^T into buffer g % 3 once P V_{g-3}
                    // has read P_{g-3} out of it (the next phase of that
                    // S_EMPTY needs S_g itself, so the wait cannot miss it).
                    // Q (BF16 tile or E4M3 codes) in shared memory, buffer k & 1.
                    ok = mbar_wait_warp(bar(Bar::Q_FULL + (k & 1)), (k >> 1) & 1, wc);
                    const uint32_t q_tile = s_q + (k & 1) * C::TILE_BYTES;
                    for (int j = w.j0; j < w.j1 && ok; ++j, ++g) {
                        const int st = g % C::NS;
                        const int b = g % C::NSB;
                        if (g >= C::NSB)
                            ok = mbar_wait_warp(bar(Bar::S_EMPTY + b), ((g - C::NSB) / C::NSB) & 1, wc);
                        ok = ok && mbar_wait_warp(bar(Bar::K_FULL + st), (g / C::NS) & 1, wc);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t k_tile = s_k + st * C::QK_BYTES;
                        const uint32_t d_tmem = tmem + C::col_s(b);
                        if constexpr (FP8) {
                            // E4M3 codes, 32 bytes of K per instruction, both
                            // operands K-major in shared memory.
                            constexpr uint32_t id_s8 = idesc_e4m3(128, 128);
#pragma unroll
                            for (int kk = 0; kk < D / 32; ++kk) {
                                uint64_t ad, bd;
                                if constexpr (D == 128) {
                                    ad = smem_desc_sw128(q_tile + kk * 32, 16, 1024);
                                    bd = smem_desc_sw128(k_tile + kk * 32, 16, 1024);
                                } else {
                                    ad = smem_desc_sw64(q_tile + kk * 32, 512);
                                    bd = smem_desc_sw64(k_tile + kk * 32, 512);
                                }
                                if (elect_one()) mma_ss_f8(d_tmem, ad, bd, id_s8, kk > 0);
                                __syncwarp();
                            }
                        } else {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                                const uint64_t ad = smem_desc_sw128(q_tile + koff, 16, 1024);
                                const uint64_t bd = smem_desc_sw128(k_tile + koff, 16, 1024);
                                if (elect_one()) mma_ss(d_tmem, ad, bd, id_s, kk > 0);
                                __syncwarp();
                            }
                        }
                        if (elect_one()) {
                            tc_commit(bar(Bar::S_FULL + b));
                            tc_commit(bar(Bar::K_EMPTY + st));
                        }
                        __syncwarp();
                    }
                }
            }
        }
    } else {
        regs_increase<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax
        // Thread (row, h): query row `row` (TMEM lane), keys [64h, 64h+64) of
        // each tile and O columns [h d/2, (h+1) d/2).  The two warps that share
        // a lane quarter swap their partial row maxima through shared memory
        // once per tile, so both apply the same running max.
        const int wq = warp & 3;             // TMEM lane quarter of this warp
        const int h = (warp - 4) >> 2;       // key / O-column half
        const int row = wq * 32 + lane;      // row inside the Q tile
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t pair_bar = 1 + wq;    // named barrier of the two warps
        float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);  // [2][2][128] maxima, [2][128] sums
        int g = 0;             // tile counter across this CTA's Q tiles
        int pending_qb = -1;   // store thread: Q buffer whose O store may still be reading it
        // Tile k from the queue; all eight warps agree on it (or on stopping).
        auto take = [&](int k) -> int {
            const int slot = k % C::QUEUE;
            const bool okq = __all_sync(
                0xffffffffu, mbar_wait(bar(Bar::ITEM_FULL + slot), (k / C::QUEUE) & 1, wc));
            const int item = okq ? items[slot] : -1;
            __syncwarp();
            if (okq && lane == 0) mbar_arrive(bar(Bar::ITEM_EMPTY + slot));
            return named_bar_and(5, 256, okq && item >= 0) ? item : -1;
        };
        int item = take(0);
        bool q_ok = item >= 0;
        for (int k = 0; item >= 0; ++k) {
            const Work w = work_of(item);
            const int qt = w.qt;
            const int bh = w.bh;
            const int grow = qt * C::BM + row;  // query index inside the head
            const int qb = k & 1;
            const uint32_t q_buf = C::OFF_Q + qb * C::TILE_BYTES;
            bool ok = q_ok;

            float m_run = -INFINITY;  // running max, base-2 units of scale * S
            float l_run = 0.f;        // this half's running sum of 2^(x - m_run)
            // FP8: S holds code products; Q's tile scale (and below K's) turn
            // them into scores.
            const float c_q = FP8 ? scale_log2 * q_scale[static_cast<long long>(bh) * n_tiles + qt]
                                  : scale_log2;
            const int bkv = (bh / Hq) * (Hq / n_rep) + (bh % Hq) / n_rep;
            for (int j = w.j0; j < w.j1; ++j, ++g) {
                const int b = g % C::NSB;
                // Factor from S to base-2 exponents for this key tile (at
                // least FLT_MIN, so that masked entries stay -inf).
                const float c_s =
                    FP8 ? fmaxf(c_q * k_scale[static_cast<long long>(bkv) * n_kv_tiles + j],
                                1.17549435e-38f)
                        : scale_log2;
                const uint32_t t_s = t_lane + C::col_s(b) + 64 * h;
                // A failed wait is carried to the pair barrier rather than
                // breaking here, so that both warps leave the loop together.
                const bool okw = ok && __all_sync(0xffffffffu,
                                                  mbar_wait(bar(Bar::S_FULL + b), (g / C::NSB) & 1, wc));
                float s[64];
                float mx = -INFINITY;
                if (okw) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t r[32];
                        tmem_ld32(t_s + c * 32, r);
#pragma unroll
                        for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[e]);
                    }
                    const int key0 = j * C::BN + 64 * h;  // key index of entry 0
                    if ((CAUSAL && j == qt) || key0 + 64 > Nk) {
                        // Keys past the row (causal) or past Nk: entry c is
                        // kept while c < lim.
                        const int lim = (CAUSAL ? min(grow + 1, Nk) : Nk) - key0;
#pragma unroll
                        for (int c = 0; c < 64; ++c) s[c] = c < lim ? s[c] : -INFINITY;
                    }
                    // Four independent running maxima, then their max: a chain
                    // of 8 three-input max instructions instead of 32.
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < 64; c += 8)
#pragma unroll
                        for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], s[c + 2 * u], s[c + 2 * u + 1]);
                    mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
                }
                xch[((g & 1) * 2 + h) * 128 + row] = mx;
                ok = named_bar_and(pair_bar, 64, okw);
                if (!ok) break;
                const float m_tile = fmaxf(mx, xch[((g & 1) * 2 + (h ^ 1)) * 128 + row]) * c_s;
                const bool rescale = m_tile > m_run + 8.0f;
                float alpha = 1.f;
                if (rescale) {
                    alpha = ex2_approx(m_run - m_tile);
                    m_run = m_tile;
                }
                const float2 c_s2 = make_float2(c_s, c_s);
                const float2 neg_m2 = make_float2(-m_run, -m_run);
                float2 sum2 = make_float2(0.f, 0.f);  // even and odd keys
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float2 x = fma2(make_float2(s[2 * e], s[2 * e + 1]), c_s2, neg_m2);
                    const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    sum2 = add2(sum2, pp);
                    pk[e] = pack_bf16x2(pp.x, pp.y);
                }
                const float sum = sum2.x + sum2.y;
                l_run = l_run * alpha + sum;
                const bool any_rescale = __any_sync(0xffffffffu, rescale) && j > w.j0;
                if (any_rescale) {
                    // A rescale of O needs PV_{j-1} to have run (O then holds
                    // the sum up to it): its commit frees the previous S buffer.
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::S_EMPTY + (g - 1) % C::NSB),
                                                           ((g - 1) / C::NSB) & 1, wc));
                    if (!ok) continue;  // the next pair barrier (or the loop end) reports it
                    tc_fence_after();
                }
                // P (BF16) over this thread's scores, already in registers:
                // keys [64h, 64h+64) at columns [64h, 64h+32) of S buffer b.
                tmem_st32(t_s, pk);
                if (any_rescale) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t r[32];
                        const uint32_t t_o = t_lane + C::COL_O + (D / 2) * h + c * 32;
                        tmem_ld32(t_o, r);
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 v = mul2(make_float2(__uint_as_float(r[e]),
                                                              __uint_as_float(r[e + 1])), a2);
                            r[e] = __float_as_uint(v.x);
                            r[e + 1] = __float_as_uint(v.y);
                        }
                        tmem_st32(t_o, r);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Bar::P_FULL + b));
                if (j == w.j0 && threadIdx.x == kStoreThread && pending_qb >= 0) {
                    // The previous tile's O store has had a whole tile of time:
                    // wait for it to finish reading its Q buffer, then free it.
                    bulk_wait_read_all();
                    mbar_arrive(bar(Bar::Q_EMPTY + pending_qb));
                    pending_qb = -1;
                }
            }
            // The next tile is taken before this tile's epilogue; its first
            // score MMAs (Q from shared memory) run meanwhile.
            const int next = take(k + 1);
            q_ok = next >= 0;
            // Both warps of the pair reach this barrier after the same iteration.
            xch[512 + h * 128 + row] = l_run;
            ok = named_bar_and(pair_bar, 64, ok);
            const float l_tot = l_run + xch[512 + (h ^ 1) * 128 + row];
            if (ok)  // the tile's last P V has run
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::S_EMPTY + (g - 1) % C::NSB),
                                                       ((g - 1) / C::NSB) & 1, wc));
            if (ok) {
                tc_fence_after();
                const float inv_l = 1.f / l_tot;
                const float lse_row = (m_run + lg2_approx(l_tot)) * 0.69314718055994531f;
                if constexpr (SPLIT) {
                    // Partial of this key chunk: O / l and LSE in FP32, merged
                    // later.  The TMEM loads are warp-wide; only real rows store.
                    const long long prow = (static_cast<long long>(w.s) * BH + bh) * N + grow;
                    if (h == 0 && grow < N) lse_part[prow] = lse_row;
                    float4* dst = reinterpret_cast<float4*>(o_part + prow * D + (D / 2) * h);
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(t_lane + C::COL_O + (D / 2) * h + cc * 32, r);
                        if (grow < N) {
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                dst[cc * 8 + u] = make_float4(
                                    __uint_as_float(r[4 * u]) * inv_l,
                                    __uint_as_float(r[4 * u + 1]) * inv_l,
                                    __uint_as_float(r[4 * u + 2]) * inv_l,
                                    __uint_as_float(r[4 * u + 3]) * inv_l);
                        }
                    }
                } else {
                    if (h == 0 && grow < N) lse[static_cast<long long>(bh) * N + grow] = lse_row;
                    // O / l -> bf16 into this tile's Q buffer (its score MMAs are done),
                    // in the TMA box layout: this half's d/2 columns are
                    // 32-column chunks h d/64 ... .
                    uint8_t* stage = smem + q_buf;
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc) {
                        const int c = h * (D / 64) + cc;  // 32-column chunk of the row
                        uint32_t r[32];
                        tmem_ld32(t_lane + C::COL_O + c * 32, r);
                        const int box = c >> 1;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            uint4 pkd;
                            pkd.x = pack_bf16x2(__uint_as_float(r[8 * u + 0]) * inv_l,
                                                __uint_as_float(r[8 * u + 1]) * inv_l);
                            pkd.y = pack_bf16x2(__uint_as_float(r[8 * u + 2]) * inv_l,
                                                __uint_as_float(r[8 * u + 3]) * inv_l);
                            pkd.z = pack_bf16x2(__uint_as_float(r[8 * u + 4]) * inv_l,
                                                __uint_as_float(r[8 * u + 5]) * inv_l);
                            pkd.w = pack_bf16x2(__uint_as_float(r[8 * u + 6]) * inv_l,
                                                __uint_as_float(r[8 * u + 7]) * inv_l);
                            const int chunk = ((c & 1) * 4 + u) ^ (row & 7);
                            *reinterpret_cast<uint4*>(stage + box * C::BOX_BYTES + row * 128 +
                                                      chunk * 16) = pkd;
                        }
                    }
                }
                fence_async_smem();
            }
            // The O columns have been read (the next tile's first PV may
            // overwrite them once its P is released), and every warp agrees on
            // whether to go on.
            if (!named_bar_and(5, 256, ok && !*abort_flag)) break;
            if (threadIdx.x == kStoreThread) {
                // (SPLIT: no store; the Q buffer is released all the same.)
                for (int kb = 0; kb < C::KB && !SPLIT; ++kb)
                    tma_store_3d(&tm_o, s_q + qb * C::TILE_BYTES + kb * C::BOX_BYTES, kb * 64,
                                 qt * C::BM, bh);
                bulk_commit();
                pending_qb = qb;
            }
            item = next;
        }
        if (threadIdx.x == kStoreThread && pending_qb >= 0) bulk_wait_read_all();
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    // The commits come from the lane that issued each warp's MMAs.
    if (warp == 2 && elect_one()) tc_commit(bar(Bar::DONE));
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

template <int D, bool CAUSAL, bool SPLIT, bool FP8 = false>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
    using C = FwdCfg<D, FP8>;
    auto kern = fwd_bf16_kernel<D, CAUSAL, SPLIT, FP8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.N + C::BM - 1) / C::BM;
    const int group = claim_group(n_tiles, CAUSAL);
    const long long n_items = static_cast<long long>(a.B) * a.H * n_tiles * a.n_splits;
    const int grid = static_cast<int>(n_items < a.num_sms ? n_items : a.num_sms);
    e = launch_overlapped(
        kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, *a.tm_q, *a.tm_k, *a.tm_v,
        *a.tm_o, a.lse, a.N, a.B * a.H, a.H, a.H / a.Hkv, n_tiles, group, a.scale_log2, a.status,
        a.timeout_ns, a.work, a.Nk, a.n_splits, a.chunk_tiles, a.o_part, a.lse_part, a.q_scale,
        a.k_scale);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_fwd_t<64, true, false>(a, stream)
                                   : launch_fwd_t<64, false, false>(a, stream);
    return a.causal ? launch_fwd_t<128, true, false>(a, stream)
                    : launch_fwd_t<128, false, false>(a, stream);
}

cudaError_t launch_fwd_splitkv_bf16(const FwdArgs& a, cudaStream_t stream) {
    return a.d == 64 ? launch_fwd_t<64, false, true>(a, stream)
                     : launch_fwd_t<128, false, true>(a, stream);
}

cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_fwd_t<64, true, false, true>(a, stream)
                                   : launch_fwd_t<64, false, false, true>(a, stream);
    return a.causal ? launch_fwd_t<128, true, false, true>(a, stream)
                    : launch_fwd_t<128, false, false, true>(a, stream);
}

}  // namespace fa
