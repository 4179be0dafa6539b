// bwd_bf16_sm103.cu - attention backward, dK/dV kernel, BF16 in / FP32
// accumulate, tcgen05 + TMEM + TMA on sm_103a.
//
// Method.  The gradient of O = softmax(scale Q K^T) V with the probabilities
// recomputed from the saved LSE instead of read back ("Flash Attention:
// Revolutionizing Transformer Efficiency", section "The Flash Attention
// algorithm", idea 2, recomputation).  Per (b, h), with D_i = dO_i . O_i:
//   P   = exp(scale S - LSE)      dV = P^T dO        dP = dO V^T
//   dS  = P o (dP - D)            dK = scale dS^T Q  (dQ: bwd_dq_sm103.cu)
// A work item is one 128-key tile j of one K/V head: K_j and V_j stay in
// shared memory and dK_j, dV_j in TMEM while the item loops over the 128-row
// Q tiles i that see those keys (i >= j when causal) of every query head that
// reads this K/V head (one head in multi-head attention, the group in
// grouped-query attention).  The parallelism over key tiles is the sequence
// parallelism of "FlashAttention-2" (technical architecture, improvement 2);
// dQ is left to a second kernel, so nothing here is reduced across CTAs.
//
// GB300 mapping: a persistent kernel, one CTA per SM (512 threads), that
// claims key tiles from a per-launch counter (heavy tiles first, a few heads
// at a time so that their Q and dO tiles stay in L2).  Items run back to back:
// the next item's K, V and first [Q | dO] stages load while the current one
// finishes, and a warpgroup of its own writes the finished dK, dV out of TMEM
// while the next item computes.
//   warp 0      TMA producer: K_j per item once issuer A's last S^T of the
//               previous item has finished, then the item's first [Q_i | dO_i]
//               stage, then V_j once issuer B's last dP^T has; per Q tile, a
//               two-deep ring of [Q_i | dO_i] stages plus the 128-entry LSE2 /
//               D vectors.
//   warps 1, 2  two MMA issuers (whole warps; one elected lane issues), so
//               that one keeps the pipe fed while the other waits.  Each
//               issuer overwrites only TMEM it alone reads, after those reads
//               in its own issue order:
//                 issuer A: dV += P^T_t dO_t (A = P^T in TMEM, after P_FULL),
//                           then S^T_t+1 = K Q_t+1^T over P^T_t;
//                 issuer B: dK += dS^T_t Q_t (A = dS^T in TMEM, after DS_FULL),
//                           then dP^T_t+1 = V dO_t+1^T over dS^T_t.
//               An item's first dV (dK) MMA, which overwrites the
//               accumulator, waits until the epilogue warps have read the
//               previous item's dV (dK) out.
//   warp 3      claims key tiles (the next one once the producer has issued
//               the current one's last loads) into a small queue that every
//               role reads in order.
//   warps 4-11  thread (r, h) owns key row r (TMEM lane r) and column half h
//               (warps 4-7: h = 0, warps 8-11: h = 1).  Phase P: 64 entries of
//               the P^T row = exp2(S^T * scale*log2e - LSE2), kept in
//               registers and written back as BF16 into the first 32 of its
//               own 64 S^T columns, in two parts of 32 entries, each released
//               to issuer A on its own barrier, so that dV's products for the
//               first part run while the second is computed.  Phase dS: dS^T = P o (dP^T - D), BF16,
//               likewise into its own dP^T columns (scale is applied to dK
//               once, when it leaves TMEM).
//   warps 12-15 epilogue: warp w reads rows 32 (w % 4) .. +32 of dV, then of
//               dK, 32 columns at a time out of TMEM into a 4 KB swizzled
//               shared-memory box and writes each box by TMA store.  An SM
//               writes about 30 bytes a cycle, so the 2 x 64 KB of FP32
//               gradients of an item take thousands of cycles; here they are
//               written while the next item's tiles run.
// Warpgroups 0 and 3 hand registers to the math warpgroups 1 and 2.
// TMEM columns: S^T [0,128) (P^T halves at [0,32) and [64,96)),
// dP^T [128,256) (dS^T halves at [128,160) and [192,224)), dV [256,256+d),
// dK [256+d, 256+2d).  All waits are bounded (see sm103_primitives.cuh).
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

constexpr int kMaxDynSmem = 232448;     // 227 KB opt-in limit per block
constexpr uint32_t kRegsLight = 72;     // warpgroups 0 and 3 after the split (no spills)
constexpr uint32_t kRegsMath = 184;     // warpgroups 1 and 2 after the split
static_assert(128 * (2 * kRegsLight + 2 * kRegsMath) <= 512 * 128, "register split");

template <int D>
struct BwdCfg {
    static constexpr int BM = 128;  // query rows per Q tile
    static constexpr int BN = 128;  // keys per item
    static constexpr int KB = D / 64;
    static constexpr int BOX_BYTES = 128 * 64 * 2;      // 128 x 64 bf16
    static constexpr int TILE_BYTES = KB * BOX_BYTES;    // 128 x D bf16
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // [Q | dO]
    static constexpr int NSQ = 2;                        // stage ring depth
    static constexpr int QUEUE = 4;                      // claimed-item queue depth
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE_BYTES;
    static constexpr int OFF_STAGE = OFF_V + TILE_BYTES;
    static constexpr int OFF_VEC = OFF_STAGE + NSQ * STAGE_BYTES;  // NSQ x (lse2, delta)
    static constexpr int NBOX = 8;  // epilogue boxes of 4 KB, two per epilogue warp
    static constexpr int OFF_STG = OFF_VEC + NSQ * 1024;
    static constexpr int OFF_BAR = OFF_STG + NBOX * 4096;
    static constexpr int BAR_BYTES = 256;
    static constexpr int OFF_ITEMS = OFF_BAR + BAR_BYTES;
    static constexpr int LAYOUT_BYTES = OFF_ITEMS + QUEUE * 4;
    // Alignment slack of up to 1 KB, as much as the limit leaves (the dynamic
    // window starts 1024-byte aligned in practice; the kernel checks).
    static constexpr int SMEM_BYTES =
        (LAYOUT_BYTES + 1024 <= kMaxDynSmem) ? LAYOUT_BYTES + 1024 : kMaxDynSmem;
    static_assert(LAYOUT_BYTES <= kMaxDynSmem, "backward tiles do not fit in shared memory");
    static_assert(OFF_STG % 1024 == 0, "swizzled staging boxes need 1024-byte alignment");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D;
    static constexpr int THREADS = 512;
    static constexpr int COMPUTE_WARPS = 8;
    // Arrivals on ITEM_EMPTY: producer, two issuers, 8 math and 4 epilogue warps.
    static constexpr int ITEM_READERS = 15;
};

template <int NSQ, int QUEUE>
struct BwdBars {
    // K and V are reloaded separately: K is free once issuer A's last S^T
    // of an item has finished, V once issuer B's last dP^T has, about one
    // MMA group later.
    static constexpr int K_FULL = 0;
    static constexpr int V_FULL = K_FULL + 1;
    static constexpr int K_EMPTY = V_FULL + 1;
    static constexpr int V_EMPTY = K_EMPTY + 1;
    // A stage holds Q (with LSE2 and D) and dO, each with its own barriers:
    // dO is last read by issuer A's dV, about one MMA group before Q's last
    // reader, issuer B's dK, so the next dO loads that much earlier and Q's
    // load, on the path to the next S^T, moves half the bytes.
    static constexpr int Q_FULL = V_EMPTY + 1;
    static constexpr int Q_EMPTY = Q_FULL + NSQ;   // S^T (A) and dK (B) done
    static constexpr int DO_FULL = Q_EMPTY + NSQ;
    static constexpr int DO_EMPTY = DO_FULL + NSQ;  // dP^T (B) and dV (A) done
    static constexpr int S_FULL = DO_EMPTY + NSQ;
    static constexpr int DP_FULL = S_FULL + 1;
    // P^T is released in two parts (queries 0-31 and 64-95, then 32-63 and
    // 96-127), so that dV's first four products start while the second part
    // is computed.
    static constexpr int P_FULL = DP_FULL + 1;
    static constexpr int P_FULL2 = P_FULL + 1;
    static constexpr int DS_FULL = P_FULL2 + 1;
    static constexpr int ACC_FULL = DS_FULL + 1;
    static constexpr int DV_FREE = ACC_FULL + 1;
    static constexpr int DK_FREE = DV_FREE + 1;
    static constexpr int ITEM_FULL = DK_FREE + 1;  // QUEUE
    static constexpr int ITEM_EMPTY = ITEM_FULL + QUEUE;
    static constexpr int CLAIM_OK = ITEM_EMPTY + QUEUE;
    static constexpr int DONE = CLAIM_OK + 1;
    static constexpr int COUNT = DONE + 1;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(512, 1)
    bwd_dkdv_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk,
                         const __grid_constant__ CUtensorMap tm_dv,
                         const float* __restrict__ delta, const float* __restrict__ lse2,
                         int N, int n_pad, int BHkv, int Hkv, int n_rep, int n_tiles,
                         int group, float scale, float scale_log2, unsigned int* status,
                         unsigned long long timeout_ns, unsigned int* work) {
    using C = BwdCfg<D>;
    using Bar = BwdBars<C::NSQ, C::QUEUE>;
    static_assert(8 * Bar::COUNT + 8 <= C::BAR_BYTES, "barrier area");
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
    volatile int* items = reinterpret_cast<volatile int*>(smem + C::OFF_ITEMS);
    const int n_items = BHkv * n_tiles;

    // Item: key tile kt of K/V head bkv (key tile 0 sees every Q tile under a
    // causal mask: heavy tiles first, a few heads at a time).  Step t of an
    // item covers query head bhq0 + t / n_q of the K/V head's group (Hq =
    // n_rep * Hkv) and its Q tile i0 + t % n_q.
    struct Work {
        int kt, bkv, i0, n_q, n_steps, bhq0;
    };
    auto work_of = [&](int item) -> Work {
        const TileHead th = grouped_order(item, BHkv, n_tiles, group, false);
        Work w;
        w.kt = th.tile;
        w.bkv = th.head;
        w.i0 = CAUSAL ? w.kt : 0;
        w.n_q = n_tiles - w.i0;
        w.n_steps = n_rep * w.n_q;
        w.bhq0 = (w.bkv / Hkv) * (Hkv * n_rep) + (w.bkv % Hkv) * n_rep;
        return w;
    };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(Bar::K_FULL), 1);
        mbar_init(bar(Bar::V_FULL), 1);
        mbar_init(bar(Bar::K_EMPTY), 1);  // issuer A's last S^T of the item
        mbar_init(bar(Bar::V_EMPTY), 1);  // issuer B's last dP^T of the item
        for (int s = 0; s < C::NSQ; ++s) {
            mbar_init(bar(Bar::Q_FULL + s), 1);
            mbar_init(bar(Bar::Q_EMPTY + s), 2);  // one commit per issuer
            mbar_init(bar(Bar::DO_FULL + s), 1);
            mbar_init(bar(Bar::DO_EMPTY + s), 2);
        }
        mbar_init(bar(Bar::S_FULL), 1);
        mbar_init(bar(Bar::DP_FULL), 1);
        mbar_init(bar(Bar::P_FULL), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::P_FULL2), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::DS_FULL), C::COMPUTE_WARPS);
        mbar_init(bar(Bar::ACC_FULL), 2);
        mbar_init(bar(Bar::DV_FREE), 4);  // one arrival per epilogue warp
        mbar_init(bar(Bar::DK_FREE), 4);
        for (int i = 0; i < C::QUEUE; ++i) {
            mbar_init(bar(Bar::ITEM_FULL + i), 1);
            mbar_init(bar(Bar::ITEM_EMPTY + i), C::ITEM_READERS);
        }
        mbar_init(bar(Bar::CLAIM_OK), 1);
        mbar_init(bar(Bar::DONE), 2);
        *abort_flag = 0;
        mbar_fence_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_do);
        prefetch_tensormap(&tm_dk);
        prefetch_tensormap(&tm_dv);
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

    // Item k of this CTA from the queue (single-thread roles); -1 at the end
    // of the work or when a wait gave up.
    auto take_item = [&](int k) -> int {
        const int slot = k % C::QUEUE;
        if (!mbar_wait(bar(Bar::ITEM_FULL + slot), (k / C::QUEUE) & 1, wc)) return -1;
        const int item = items[slot];
        mbar_arrive(bar(Bar::ITEM_EMPTY + slot));
        return item;
    };
    // The same for a whole warp: every lane waits and reads, lane 0 arrives.
    auto take_item_warp = [&](int k) -> int {
        const int slot = k % C::QUEUE;
        const bool ok = __all_sync(
            0xffffffffu, mbar_wait(bar(Bar::ITEM_FULL + slot), (k / C::QUEUE) & 1, wc));
        const int item = ok ? items[slot] : -1;
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(bar(Bar::ITEM_EMPTY + slot));
        return item;
    };

    if (warp < 4 || warp >= 12) {
        regs_decrease<kRegsLight>();
        if (warp == 3) {
            // ------------------------------------------------------------ claimer
            if (lane == 0) {
                bool ok = true, claimed_last = false;
                for (int k = 0; ok; ++k) {
                    const int slot = k % C::QUEUE;
                    if (k >= 1) ok = mbar_wait(bar(Bar::CLAIM_OK), (k - 1) & 1, wc);
                    if (ok && k >= C::QUEUE)
                        ok = mbar_wait(bar(Bar::ITEM_EMPTY + slot), ((k / C::QUEUE) - 1) & 1, wc);
                    if (!ok) break;
                    int item = static_cast<int>(blockIdx.x);
                    if (k > 0) {
                        const unsigned int t = atomicAdd(work, 1u);
                        item = static_cast<int>(gridDim.x + t);
                        if (item >= n_items) {
                            claimed_last = true;
                            // Every CTA ends with exactly one failed claim; the one
                            // that draws the last number resets the counter.
                            if (t == static_cast<unsigned int>(n_items) - 1u) atomicExch(work, 0u);
                        }
                    }
                    if (item >= n_items) item = -1;
                    items[slot] = item;
                    mbar_arrive(bar(Bar::ITEM_FULL + slot));
                    if (item < 0) break;
                }
                while (!claimed_last) {  // after giving up: finish drawing as normal
                    const unsigned int t = atomicAdd(work, 1u);
                    if (gridDim.x + t >= static_cast<unsigned int>(n_items)) {
                        claimed_last = true;
                        if (t == static_cast<unsigned int>(n_items) - 1u) atomicExch(work, 0u);
                    }
                }
            }
            __syncwarp();
        } else if (warp == 0) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                int g = 0, issued = 0, issued_do = 0, k_loads = 0, v_loads = 0;
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    const int item = take_item(k);
                    if (item < 0) break;
                    const Work w = work_of(item);
                    // K of this item once issuer A's last S^T of the previous
                    // item has finished; V (below, after the item's first
                    // [Q | dO] stage) once issuer B's last dP^T has.
                    if (k >= 1) ok = mbar_wait(bar(Bar::K_EMPTY), (k - 1) & 1, wc);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(Bar::K_FULL), C::TILE_BYTES);
                    for (int kb = 0; kb < C::KB; ++kb)
                        tma_load_3d(s_k + kb * C::BOX_BYTES, &tm_k, bar(Bar::K_FULL), kb * 64,
                                    w.kt * C::BN, w.bkv);
                    k_loads = k + 1;
                    for (int t = 0; t < w.n_steps && ok; ++t, ++g) {
                        const int st = g % C::NSQ;
                        const int use = g / C::NSQ;
                        const int i = w.i0 + t % w.n_q;
                        const int bh = w.bhq0 + t / w.n_q;  // query head
                        const long long voff = static_cast<long long>(bh) * n_pad + i * C::BM;
                        // dO first: its half of the stage frees first.
                        if (use > 0) ok = mbar_wait(bar(Bar::DO_EMPTY + st), (use - 1) & 1, wc);
                        if (!ok) break;
                        const uint32_t fo = bar(Bar::DO_FULL + st);
                        mbar_arrive_expect_tx(fo, C::TILE_BYTES);
                        for (int kb = 0; kb < C::KB; ++kb)
                            tma_load_3d(do_of(st) + kb * C::BOX_BYTES, &tm_do, fo, kb * 64,
                                        i * C::BM, bh);
                        issued_do = g + 1;
                        // Q with LSE2 and D: the math warps read D in the dS
                        // phase, which dK (Q's last reader) follows, while dV
                        // (dO's last reader) may end before it.
                        if (use > 0) ok = mbar_wait(bar(Bar::Q_EMPTY + st), (use - 1) & 1, wc);
                        if (!ok) break;
                        const uint32_t fb = bar(Bar::Q_FULL + st);
                        mbar_arrive_expect_tx(fb, C::TILE_BYTES + 1024);
                        for (int kb = 0; kb < C::KB; ++kb)
                            tma_load_3d(q_of(st) + kb * C::BOX_BYTES, &tm_q, fb, kb * 64,
                                        i * C::BM, bh);
                        bulk_load(s_vec + st * 1024, lse2 + voff, 512, fb);
                        bulk_load(s_vec + st * 1024 + 512, delta + voff, 512, fb);
                        issued = g + 1;
                        if (t == 0) {
                            if (k >= 1) ok = mbar_wait(bar(Bar::V_EMPTY), (k - 1) & 1, wc);
                            if (!ok) break;
                            mbar_arrive_expect_tx(bar(Bar::V_FULL), C::TILE_BYTES);
                            for (int kb = 0; kb < C::KB; ++kb)
                                tma_load_3d(s_v + kb * C::BOX_BYTES, &tm_v, bar(Bar::V_FULL),
                                            kb * 64, w.kt * C::BN, w.bkv);
                            v_loads = k + 1;
                        }
                    }
                    if (ok) mbar_arrive(bar(Bar::CLAIM_OK));  // the next item may be claimed
                }
                // Drain: no copy may still be landing when the CTA exits.
                if (k_loads > 0)
                    mbar_wait_drain(bar(Bar::K_FULL), (k_loads - 1) & 1, timeout_ns);
                if (v_loads > 0)
                    mbar_wait_drain(bar(Bar::V_FULL), (v_loads - 1) & 1, timeout_ns);
                for (int t = (issued_do > C::NSQ ? issued_do - C::NSQ : 0); t < issued_do; ++t)
                    mbar_wait_drain(bar(Bar::DO_FULL + t % C::NSQ), (t / C::NSQ) & 1, timeout_ns);
                for (int t = (issued > C::NSQ ? issued - C::NSQ : 0); t < issued; ++t)
                    mbar_wait_drain(bar(Bar::Q_FULL + t % C::NSQ), (t / C::NSQ) & 1, timeout_ns);
            }
            __syncwarp();
        } else if (warp == 1 || warp == 2) {
            // ------------------------------------------------------------ MMA issuers
            // Each issuer is a whole warp: every lane waits and computes the
            // operands, one elected lane issues the MMAs and commits.
            {
                constexpr uint32_t id_sp = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
                constexpr uint32_t id_kv = idesc_bf16(128, D, 0, 1);    // dV, dK: B MN-major
                const bool issuer_a = (warp == 1);
                // Base descriptors; each MMA below only moves the start address.
                const uint64_t d_k = smem_desc_sw128(s_k, 16, 1024);  // A of S^T
                const uint64_t d_v = smem_desc_sw128(s_v, 16, 1024);  // A of dP^T
                // Stage 0 descriptors; stage st sits st * STAGE_BYTES further on.
                // issuer A: Q (K-major, B of S^T) and dO (MN-major, B of dV);
                // issuer B: dO (K-major, B of dP^T) and Q (MN-major, B of dK).
                const uint64_t d_kmaj0 = smem_desc_sw128(issuer_a ? q_of(0) : do_of(0), 16, 1024);
                const uint64_t d_mn0 =
                    smem_desc_sw128(issuer_a ? do_of(0) : q_of(0), C::BOX_BYTES, 1024);
                const uint64_t d_first = issuer_a ? d_k : d_v;
                const uint32_t c_first = issuer_a ? C::COL_S : C::COL_DP;  // S^T or dP^T
                const uint32_t c_acc = issuer_a ? C::COL_DV : C::COL_DK;   // dV or dK
                const uint32_t c_a = issuer_a ? C::COL_S : C::COL_DP;      // P^T or dS^T
                const int ready_bar = issuer_a ? Bar::P_FULL : Bar::DS_FULL;
                // Stage halves: the first GEMM's B operand (Q for A, dO for
                // B) and the accumulation's (dO for A, Q for B).
                const int first_full = issuer_a ? Bar::Q_FULL : Bar::DO_FULL;
                const int first_empty = issuer_a ? Bar::Q_EMPTY : Bar::DO_EMPTY;
                const int acc_full = issuer_a ? Bar::DO_FULL : Bar::Q_FULL;
                const int acc_empty = issuer_a ? Bar::DO_EMPTY : Bar::Q_EMPTY;
                const int full_bar = issuer_a ? Bar::S_FULL : Bar::DP_FULL;
                const int free_bar = issuer_a ? Bar::DV_FREE : Bar::DK_FREE;
                // First GEMM of step g: S^T = K Q^T (A) or dP^T = V dO^T (B).
                auto issue_first = [&](int g) -> bool {
                    const int st = g % C::NSQ;
                    if (!mbar_wait_warp(bar(first_full + st), (g / C::NSQ) & 1, wc)) return false;
                    tc_fence_after();
                    const uint64_t d_b = desc_advance(d_kmaj0, st * C::STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                        const uint64_t ad = desc_advance(d_first, koff);
                        const uint64_t bd = desc_advance(d_b, koff);
                        if (elect_one()) mma_ss(tmem + c_first, ad, bd, id_sp, kk > 0);
                        __syncwarp();
                    }
                    if (elect_one()) {
                        tc_commit(bar(full_bar));
                        tc_commit(bar(first_empty + st));  // this half of the stage is read
                    }
                    __syncwarp();
                    return true;
                };
                int g = 0;  // step counter across this CTA's items
                bool ok = true;
                for (int k = 0; ok; ++k) {
                    const int item = take_item_warp(k);
                    if (item < 0) break;
                    const Work w = work_of(item);
                    const int kv_full = issuer_a ? Bar::K_FULL : Bar::V_FULL;
                    const int kv_empty = issuer_a ? Bar::K_EMPTY : Bar::V_EMPTY;
                    ok = mbar_wait_warp(bar(kv_full), k & 1, wc) && issue_first(g);
                    // K (V) is read for the last time by the item's last first GEMM.
                    if (ok && w.n_steps == 1 && elect_one()) tc_commit(bar(kv_empty));
                    __syncwarp();
                    for (int t = 0; t < w.n_steps && ok; ++t, ++g) {
                        const int st = g % C::NSQ;
                        ok = mbar_wait_warp(bar(ready_bar), g & 1, wc);
                        // The item's first accumulation overwrites dV (dK): the
                        // epilogue must have read the previous item's out.
                        if (ok && t == 0 && k >= 1) ok = mbar_wait_warp(bar(free_bar), (k - 1) & 1, wc);
                        // The accumulation's own operand half of the stage.
                        ok = ok && mbar_wait_warp(bar(acc_full + st), (g / C::NSQ) & 1, wc);
                        // Issuer B holds dK_t and dP^T_t+1 until issuer A's S^T_t+1 is
                        // done: A's dV_t, S^T_t+1 lead to the next P phase and should
                        // not share the pipe; B's pair then runs during that P phase.
                        // S_FULL cannot pass step t+1 before this wait: S^T_t+2 needs
                        // the stage that B frees only after dK_t.
                        if (ok && !issuer_a && t + 1 < w.n_steps)
                            ok = mbar_wait_warp(bar(Bar::S_FULL), (g + 1) & 1, wc);
                        if (!ok) break;
                        tc_fence_after();
                        // dV += P^T dO (A) or dK += dS^T Q (B); the BF16 halves of
                        // P^T / dS^T (queries 0-63, 64-127) sit at columns [0,32)
                        // and [64,96) of their fp32 region.
                        const uint64_t d_mn = desc_advance(d_mn0, st * C::STAGE_BYTES);
                        // Queries 0-31 and 64-95 first (products 0, 1, 4, 5), then
                        // 32-63 and 96-127; issuer A waits for the second part of
                        // P^T in between.
#pragma unroll
                        for (int part = 0; part < 2; ++part) {
                            if (part == 1 && issuer_a) {
                                ok = mbar_wait_warp(bar(Bar::P_FULL2), g & 1, wc);
                                if (!ok) break;
                                tc_fence_after();
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int kk = (u < 2 ? u : u + 2) + 2 * part;
                                const uint32_t acol = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
                                const uint64_t bd = desc_advance(d_mn, kk * 2048);
                                if (elect_one())
                                    mma_ts(tmem + c_acc, tmem + c_a + acol, bd, id_kv,
                                           (t > 0 || kk > 0) ? 1u : 0u);
                                __syncwarp();
                            }
                        }
                        if (!ok) break;
                        // This issuer no longer reads stage g.
                        if (elect_one()) tc_commit(bar(acc_empty + st));
                        __syncwarp();
                        if (t + 1 < w.n_steps) {
                            ok = issue_first(g + 1);
                            if (ok && t + 2 == w.n_steps && elect_one()) tc_commit(bar(kv_empty));
                            __syncwarp();
                        }
                    }
                    if (ok && elect_one()) tc_commit(bar(Bar::ACC_FULL));
                    __syncwarp();
                }
            }
        } else {
            // ------------------------------------------------------------ epilogue
            // Warp e (of warps 12-15) owns TMEM lanes 32 (e % 4) .. +32: rows
            // of dV, then of dK, 32 columns (one 4 KB box) at a time, through
            // two boxes in turn.  A box is rewritten once the store issued
            // from it two chunks earlier has read it, so the reads out of
            // TMEM run a chunk ahead of the SM's write path and each
            // accumulator is released that much sooner.
            const int wq = warp & 3;
            const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
            const uint32_t box0 = s_base + C::OFF_STG + static_cast<uint32_t>(wq * 2 * 4096);
            constexpr int NCH = D / 32;  // 32-column chunks of dV (and of dK)
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int item = take_item_warp(k);
                if (item < 0) break;
                const Work w = work_of(item);
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::ACC_FULL), k & 1, wc));
                if (!ok) break;
                tc_fence_after();
                const int row0 = w.kt * C::BN + wq * 32;
#pragma unroll 1
                for (int c = 0; c < 2 * NCH; ++c) {
                    uint32_t a[32];
                    tmem_ld32(t_lane + C::COL_DV + 32 * c, a);  // dK follows dV
                    if (c == NCH - 1 || c == 2 * NCH - 1) {
                        // This warp has read its rows of dV (dK) out.
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(c == NCH - 1 ? Bar::DV_FREE : Bar::DK_FREE));
                    }
                    // Every chunk commits one group (empty past N), so "at
                    // most one group still reading" frees this chunk's box.
                    if (lane == 0) bulk_wait_read_allow1();
                    __syncwarp();
                    const uint32_t box = box0 + static_cast<uint32_t>((c & 1) * 4096);
                    st_row_sw128_f32(box, lane, a, c < NCH ? 1.f : scale);
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (row0 < N)
                            tma_store_3d(c < NCH ? &tm_dv : &tm_dk, box, 32 * (c % NCH), row0,
                                         w.bkv);
                        bulk_commit();
                    }
                }
            }
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
        }
    } else {
        regs_increase<kRegsMath>();
        // ------------------------------------------------------------ P / dS
        const int wq = warp & 3;
        const int h = (warp - 4) >> 2;       // column half
        const int r = wq * 32 + lane;        // key row
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float* vec_base = reinterpret_cast<const float*>(smem + C::OFF_VEC);
        int g = 0;  // step counter across this CTA's items
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = take_item_warp(k);
            if (item < 0) break;
            const Work w = work_of(item);
            const int kglob = w.kt * C::BN + r;  // key index inside the head
            const bool key_pad = kglob >= N;
            for (int t = 0; t < w.n_steps; ++t, ++g) {
                const int st = g % C::NSQ;
                const int i = w.i0 + t % w.n_q;
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::S_FULL), g & 1, wc) &&
                                                 mbar_wait(bar(Bar::Q_FULL + st),
                                                           (g / C::NSQ) & 1, wc));
                if (!ok) break;
                tc_fence_after();
                const float* l2v = vec_base + st * 256 + 64 * h;
                const float* dlt = vec_base + st * 256 + 128 + 64 * h;
                // Phase P: entries [64h, 64h+64) of this key's row of P^T, in
                // two parts of 32; part q's BF16 pairs go over score columns
                // [64h + 16q, 64h + 16q + 16), already loaded.
                float p[64];
                const int q0 = i * C::BM + 64 * h;  // query index of entry 0
                const float2 c2 = make_float2(scale_log2, scale_log2);
                const float4* l2v4 = reinterpret_cast<const float4*>(l2v);  // 16-byte broadcasts
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    uint32_t sr[32];
                    tmem_ld32(t_lane + C::COL_S + 64 * h + 32 * part, sr);
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 l = l2v4[(32 * part + c) / 4];
                        const float2 x0 = fma2(make_float2(__uint_as_float(sr[c]),
                                                           __uint_as_float(sr[c + 1])),
                                               c2, make_float2(-l.x, -l.y));
                        const float2 x1 = fma2(make_float2(__uint_as_float(sr[c + 2]),
                                                           __uint_as_float(sr[c + 3])),
                                               c2, make_float2(-l.z, -l.w));
                        p[32 * part + c] = ex2_approx(x0.x);
                        p[32 * part + c + 1] = ex2_approx(x0.y);
                        p[32 * part + c + 2] = ex2_approx(x1.x);
                        p[32 * part + c + 3] = ex2_approx(x1.y);
                    }
                    if (key_pad || (CAUSAL && i == w.kt)) {
                        // Queries before the key (causal), or every query of a
                        // padding key: entry c is zeroed while c < lim.
                        const int lim = key_pad ? 64 : kglob - q0;
#pragma unroll
                        for (int c = 32 * part; c < 32 * part + 32; ++c) p[c] = c < lim ? 0.f : p[c];
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(p[32 * part + 2 * e], p[32 * part + 2 * e + 1]);
                    tmem_st16(t_lane + C::COL_S + 64 * h + 16 * part, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(part == 0 ? Bar::P_FULL : Bar::P_FULL2));
                }

                // Phase dS: dS^T = P o (dP^T - D), BF16, over its dP^T columns.
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::DP_FULL), g & 1, wc));
                if (!ok) break;
                tc_fence_after();
                {
                    uint32_t dr[64];
                    tmem_ld64(t_lane + C::COL_DP + 64 * h, dr);
                    uint32_t wv[32];
                    const float2 m1 = make_float2(-1.f, -1.f);
                    const float4* dlt4 = reinterpret_cast<const float4*>(dlt);  // 16-byte broadcasts
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int c = 2 * e;
                        const float4 dd = dlt4[c / 4];
                        // dP - D exactly as a subtraction (D * -1 is exact), then P o (dP - D).
                        const float2 t0 = fma2(make_float2(dd.x, dd.y), m1,
                                               make_float2(__uint_as_float(dr[c]),
                                                           __uint_as_float(dr[c + 1])));
                        const float2 t1 = fma2(make_float2(dd.z, dd.w), m1,
                                               make_float2(__uint_as_float(dr[c + 2]),
                                                           __uint_as_float(dr[c + 3])));
                        const float2 ds0 = mul2(make_float2(p[c], p[c + 1]), t0);
                        const float2 ds1 = mul2(make_float2(p[c + 2], p[c + 3]), t1);
                        wv[e] = pack_bf16x2(ds0.x, ds0.y);
                        wv[e + 1] = pack_bf16x2(ds1.x, ds1.y);
                    }
                    tmem_st32(t_lane + C::COL_DP + 64 * h, wv);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Bar::DS_FULL));
            }
        }
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

template <int D, bool CAUSAL>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t stream) {
    using C = BwdCfg<D>;
    auto kern = bwd_dkdv_bf16_kernel<D, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.N + C::BN - 1) / C::BN;
    const int group = claim_group(n_tiles, CAUSAL);
    const long long n_items = static_cast<long long>(a.B) * a.Hkv * n_tiles;
    const int grid = static_cast<int>(n_items < a.num_sms ? n_items : a.num_sms);
    e = launch_overlapped(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, *a.tm_q,
                          *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dk, *a.tm_dv, a.delta, a.lse2, a.N,
                          a.n_pad, a.B * a.Hkv, a.Hkv, a.H / a.Hkv, n_tiles, group, a.scale,
                          a.scale_log2, a.status, a.timeout_ns, a.work);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_bf16(const BwdArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
    return a.causal ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
}

}  // namespace fa
