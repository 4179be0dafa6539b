// fwd_bf16_sm103.cu - exact attention forward, BF16 in / FP32 accumulate,
// tcgen05 + TMEM + TMA on sm_103a.
//
// Method.  The online softmax of "LLM part 06: FlashAttention - GPU SRAM,
// tiling and online softmax" (section 2): each query row keeps a running max m
// and running sum l while key blocks stream past, and the output accumulator
// is rescaled by exp(m_old - m_new) whenever the max moves.  Loop order and
// parallelism follow "FlashAttention scaling, multi-GPU training and weight
// quantization" (section 1): one CTA per 128-row Q tile of one (batch, head),
// the K/V tiles in the inner loop, TMA copies issued by a producer warp, and
// the division by l deferred to the end ("FlashAttention-2", technical
// architecture, improvement 1).
//
// GB300 mapping (one CTA per SM, 352 threads):
//   warp 0      TMA producer: Q tile once, then K_j and V_j into an NS-deep
//               shared-memory ring (128-byte swizzle, 64-column boxes).
//   warps 1, 10 two MMA issuers (one thread each).  A: S_j = Q K_j^T into one
//               of two TMEM score buffers, once the softmax warps have read
//               S_{j-2} out of it.  B: O += P_j V_j as soon as the softmax
//               warps release P_j.  Both take A from TMEM (Q, copied there
//               once, and P), so consecutive MMAs never switch the A source,
//               which drains the tensor pipe.  One thread issues MMAs no
//               faster than the pipe runs them, so two issuers keep it fed
//               while either waits.
//   warps 2..9  softmax: thread (r, h) owns query row r (TMEM lane r) and
//               keys [64h, 64h+64) of every tile (warps 2-5: h = 0, 6-9:
//               h = 1), so two warps share each SM sub-partition's rows and
//               hide each other's latency.  First, Q row half into TMEM.  Per
//               tile: load its 64 scores (then the S buffer is free), mask,
//               swap the partial row max with the partner warp through shared
//               memory, update m and its half of l, write P as BF16 into the
//               P buffer once PV_{j-1} has read it, and rescale its
//               d/2 columns of the O accumulator only when the max grew by
//               more than 2^8 (the final O / l and LSE use the same stale
//               max, so the result is unchanged).  Epilogue: the two halves of
//               l are summed, O / l goes to BF16 through shared memory and a
//               TMA store; LSE = ln 2 * (m + log2 l).
//
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+d), Q [256+d, 256+3d/2),
// P [256+3d/2, 320+3d/2) (all 512 columns at d = 128).  All waits are
// bounded (see sm103_primitives.cuh).
#include "fa_internal.h"
#include "sm103_primitives.cuh"

namespace fa {
namespace {

template <int D>
struct FwdCfg {
    static constexpr int BM = 128;                    // query rows per CTA
    static constexpr int BN = 128;                    // keys per K/V tile
    static constexpr int KB = D / 64;                 // 64-column (128-byte) boxes per row
    static constexpr int BOX_BYTES = 128 * 64 * 2;    // one 128 x 64 bf16 box
    static constexpr int TILE_BYTES = KB * BOX_BYTES; // one 128 x D bf16 tile
    static constexpr int NS = (D == 128) ? 2 : 4;     // K/V ring depth
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int OFF_XCH = OFF_BAR + BAR_BYTES;  // row maxima and sums of the halves
    static constexpr int XCH_BYTES = 6 * 128 * 4;
    static constexpr int SMEM_BYTES = OFF_XCH + XCH_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    // S0, S1: scores (FP32); O: accumulator (FP32); Q and P: BF16 pairs, the
    // A operands of S = Q K^T and O += P V.
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
    static constexpr uint32_t COL_Q = COL_O + D, COL_P = COL_Q + D / 2;
    static_assert(COL_P + BN / 2 <= TMEM_COLS, "TMEM columns");
    static constexpr int THREADS = 352;
};

// Barrier slots (8 bytes each) inside the barrier area.
template <int NS>
struct FwdBars {
    static constexpr int Q_FULL = 0;
    static constexpr int K_FULL = 1;
    static constexpr int V_FULL = K_FULL + NS;
    static constexpr int K_EMPTY = V_FULL + NS;
    static constexpr int V_EMPTY = K_EMPTY + NS;
    static constexpr int S_FULL = V_EMPTY + NS;  // 2
    static constexpr int S_EMPTY = S_FULL + 2;   // 2
    static constexpr int QT_FULL = S_EMPTY + 2;
    static constexpr int P_FULL = QT_FULL + 1;
    static constexpr int O_FULL = P_FULL + 1;
    static constexpr int DONE = O_FULL + 1;
    static constexpr int COUNT = DONE + 1;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(352, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, float* __restrict__ lse, int N,
                    int BH, int n_tiles, int group, float scale_log2, unsigned int* status,
                    unsigned long long timeout_ns) {
    using C = FwdCfg<D>;
    using Bar = FwdBars<C::NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + C::OFF_Q;
    const uint32_t s_k = s_base + C::OFF_K;
    const uint32_t s_v = s_base + C::OFF_V;
    const uint32_t s_bar = s_base + C::OFF_BAR;
    auto bar = [&](int slot) -> uint32_t { return s_bar + 8u * static_cast<uint32_t>(slot); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * Bar::COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    // Heavy tiles first (with a causal mask the last Q tile sees the most
    // keys), a few heads at a time so that their K/V tiles stay in L2.
    const long long lin = blockIdx.x + static_cast<long long>(gridDim.x) *
                                           (blockIdx.y + static_cast<long long>(gridDim.y) *
                                                             blockIdx.z);
    const TileHead th = grouped_order(lin, BH, n_tiles, group, true);
    const int qt = th.tile;
    const int bh = th.head;
    const int n_kv = CAUSAL ? qt + 1 : n_tiles;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(Bar::Q_FULL), 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(Bar::K_FULL + s), 1);
            mbar_init(bar(Bar::V_FULL + s), 1);
            mbar_init(bar(Bar::K_EMPTY + s), 1);
            mbar_init(bar(Bar::V_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(Bar::S_FULL + b), 1);
            mbar_init(bar(Bar::S_EMPTY + b), 8);  // one arrival per softmax warp
        }
        mbar_init(bar(Bar::QT_FULL), 8);
        mbar_init(bar(Bar::P_FULL), 8);
        mbar_init(bar(Bar::O_FULL), 1);
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

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(Bar::Q_FULL), C::TILE_BYTES);
            for (int kb = 0; kb < C::KB; ++kb)
                tma_load_3d(s_q + kb * C::BOX_BYTES, &tm_q, bar(Bar::Q_FULL), kb * 64,
                            qt * C::BM, bh);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < n_kv && ok; ++j) {
                const int st = j % C::NS;
                const int use = j / C::NS;
                if (use > 0) ok = mbar_wait(bar(Bar::K_EMPTY + st), (use - 1) & 1, wc);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(Bar::K_FULL + st), C::TILE_BYTES);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_3d(s_k + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_k,
                                bar(Bar::K_FULL + st), kb * 64, j * C::BN, bh);
                if (use > 0) ok = mbar_wait(bar(Bar::V_EMPTY + st), (use - 1) & 1, wc);
                if (!ok) {
                    // K_j is in flight: wait for it before leaving.
                    mbar_wait_drain(bar(Bar::K_FULL + st), use & 1, timeout_ns);
                    break;
                }
                mbar_arrive_expect_tx(bar(Bar::V_FULL + st), C::TILE_BYTES);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_3d(s_v + st * C::TILE_BYTES + kb * C::BOX_BYTES, &tm_v,
                                bar(Bar::V_FULL + st), kb * 64, j * C::BN, bh);
                issued = j + 1;
            }
            // Drain: no copy may still be landing when the CTA exits.
            mbar_wait_drain(bar(Bar::Q_FULL), 0, timeout_ns);
            for (int j = (issued > C::NS ? issued - C::NS : 0); j < issued; ++j) {
                mbar_wait_drain(bar(Bar::K_FULL + j % C::NS), (j / C::NS) & 1, timeout_ns);
                mbar_wait_drain(bar(Bar::V_FULL + j % C::NS), (j / C::NS) & 1, timeout_ns);
            }
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------------------ MMA issuers
        // Every MMA takes its A operand from TMEM: a 128 x 128 x 16 MMA that
        // follows one with A in shared memory (or the reverse) waits for the
        // pipe to drain, which cost about a third of the tensor time.
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);  // B = K, K-major
            constexpr uint32_t id_pv = idesc_bf16(128, D, 0, 1);   // B = V, MN-major
            if (warp == 10) {
                // Issuer B: O += P_t V_t as soon as the softmax warps release P_t.
                bool ok = true;
                for (int t = 0; t < n_kv && ok; ++t) {
                    const int st = t % C::NS;
                    ok = mbar_wait(bar(Bar::P_FULL), t & 1, wc) &&
                         mbar_wait(bar(Bar::V_FULL + st), (t / C::NS) & 1, wc);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t v_tile = s_v + st * C::TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; ++kk) {
                        // V as an MN-major B operand: 16 keys = 2 atoms of 8 rows.
                        const uint64_t bd =
                            smem_desc_sw128(v_tile + kk * 2048, C::BOX_BYTES, 1024);
                        mma_ts(tmem + C::COL_O, tmem + C::COL_P + kk * 8, bd, id_pv,
                               (t > 0 || kk > 0));
                    }
                    tc_commit(bar(Bar::V_EMPTY + st));
                    tc_commit(bar(Bar::O_FULL));
                }
            } else {
                // Issuer A: S_j = Q K_j^T into buffer j & 1 once the softmax
                // warps have read S_{j-2} out of it.  The next phase of that
                // buffer's S_EMPTY needs S_j itself, so the wait cannot miss it.
                bool ok = mbar_wait(bar(Bar::QT_FULL), 0, wc);
                for (int j = 0; j < n_kv && ok; ++j) {
                    const int st = j % C::NS;
                    const int b = j & 1;
                    if (j >= 2) ok = mbar_wait(bar(Bar::S_EMPTY + b), ((j - 2) >> 1) & 1, wc);
                    ok = ok && mbar_wait(bar(Bar::K_FULL + st), (j / C::NS) & 1, wc);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t k_tile = s_k + st * C::TILE_BYTES;
                    const uint32_t d_tmem = tmem + (b ? C::COL_S1 : C::COL_S0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                        mma_ts(d_tmem, tmem + C::COL_Q + kk * 8,
                               smem_desc_sw128(k_tile + koff, 16, 1024), id_s, kk > 0);
                    }
                    tc_commit(bar(Bar::S_FULL + b));
                    tc_commit(bar(Bar::K_EMPTY + st));
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        // Thread (row, h): query row `row` (TMEM lane), keys [64h, 64h+64) of
        // each tile and O columns [h d/2, (h+1) d/2).  The two warps that share
        // a lane quarter swap their partial row maxima through shared memory
        // once per tile, so both apply the same running max.
        const int wq = warp & 3;             // TMEM lane quarter of this warp
        const int h = (warp - 2) >> 2;       // key / O-column half
        const int row = wq * 32 + lane;      // row inside the Q tile
        const int grow = qt * C::BM + row;   // query index inside the head
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t pair_bar = 1 + wq;    // named barrier of the two warps
        float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);  // [2][2][128] maxima, [2][128] sums
        float m_run = -INFINITY;  // running max, base-2 units of scale * S
        float l_run = 0.f;        // this half's running sum of 2^(x - m_run)
        // Q into TMEM as BF16 pairs (the A operand of S = Q K^T): this thread's
        // row, elements [h d/2, (h+1) d/2), read from the swizzled tile.
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::Q_FULL), 0, wc));
        if (ok) {
            uint32_t w[D / 4];
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                const int gc = h * (D / 16) + c;  // 16-byte chunk of the row
                const uint4 v = *reinterpret_cast<const uint4*>(
                    smem + C::OFF_Q + (gc >> 3) * C::BOX_BYTES + row * 128 +
                    (((gc & 7) ^ (row & 7)) << 4));
                w[4 * c] = v.x;
                w[4 * c + 1] = v.y;
                w[4 * c + 2] = v.z;
                w[4 * c + 3] = v.w;
            }
            if constexpr (D == 128) tmem_st32(t_lane + C::COL_Q + h * (D / 4), w);
            else tmem_st16(t_lane + C::COL_Q + h * (D / 4), w);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::QT_FULL));
        }
        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;
            const uint32_t t_s = t_lane + (b ? C::COL_S1 : C::COL_S0) + 64 * h;
            // A failed wait is carried to the pair barrier rather than breaking
            // here, so that both warps leave the loop at the same barrier.
            bool okw = ok && __all_sync(0xffffffffu,
                                        mbar_wait(bar(Bar::S_FULL + b), (j >> 1) & 1, wc));
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
                // S_j is in registers: its buffer may take S_{j+2}.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(Bar::S_EMPTY + b));
                const int key0 = j * C::BN + 64 * h;  // key index of entry 0
                if ((CAUSAL && j == qt) || key0 + 64 > N) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int key = key0 + c;
                        if ((CAUSAL && key > grow) || key >= N) s[c] = -INFINITY;
                    }
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) mx = fmaxf(mx, s[c]);
            }
            xch[(b * 2 + h) * 128 + row] = mx;
            ok = named_bar_and(pair_bar, 64, okw);
            if (!ok) break;
            const float m_tile = fmaxf(mx, xch[(b * 2 + (h ^ 1)) * 128 + row]) * scale_log2;
            const bool rescale = m_tile > m_run + 8.0f;
            float alpha = 1.f;
            if (rescale) {
                alpha = ex2_approx(m_run - m_tile);
                m_run = m_tile;
            }
            const float neg_m = -m_run;
            float sum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float p0 = ex2_approx(fmaf(s[2 * e], scale_log2, neg_m));
                const float p1 = ex2_approx(fmaf(s[2 * e + 1], scale_log2, neg_m));
                sum += p0 + p1;
                pk[e] = pack_bf16x2(p0, p1);
            }
            l_run = l_run * alpha + sum;
            if (j > 0) {
                // PV_{j-1} has finished: the P buffer is free, and O holds the
                // sum up to PV_{j-1}, as a rescale needs.
                ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::O_FULL), (j - 1) & 1, wc));
                if (!ok) continue;  // the next pair barrier (or the loop end) reports it
                tc_fence_after();
            }
            // P_j (BF16): keys [64h, 64h+64) at P columns [32h, 32h+32).
            tmem_st32(t_lane + C::COL_P + 32 * h, pk);
            if (__any_sync(0xffffffffu, rescale) && j > 0) {
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t r[32];
                    const uint32_t t_o = t_lane + C::COL_O + (D / 2) * h + c * 32;
                    tmem_ld32(t_o, r);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    tmem_st32(t_o, r);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(Bar::P_FULL));
        }
        // Both warps of the pair reach this barrier after the same iteration.
        xch[512 + h * 128 + row] = l_run;
        ok = named_bar_and(pair_bar, 64, ok);
        const float l_tot = l_run + xch[512 + (h ^ 1) * 128 + row];
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(Bar::O_FULL), (n_kv - 1) & 1, wc));
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l_tot;
            if (h == 0 && grow < N)
                lse[static_cast<long long>(bh) * N + grow] =
                    (m_run + lg2_approx(l_tot)) * 0.69314718055994531f;
            // O / l -> bf16 into the (now free) Q buffer, in the TMA box layout:
            // this half's d/2 columns are 32-column chunks h d/64 ... .
            uint8_t* stage = smem + C::OFF_Q;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int c = h * (D / 64) + cc;  // 32-column chunk of the row
                uint32_t r[32];
                tmem_ld32(t_lane + C::COL_O + c * 32, r);
                const int box = c >> 1;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(r[8 * u + 0]) * inv_l,
                                      __uint_as_float(r[8 * u + 1]) * inv_l);
                    w.y = pack_bf16x2(__uint_as_float(r[8 * u + 2]) * inv_l,
                                      __uint_as_float(r[8 * u + 3]) * inv_l);
                    w.z = pack_bf16x2(__uint_as_float(r[8 * u + 4]) * inv_l,
                                      __uint_as_float(r[8 * u + 5]) * inv_l);
                    w.w = pack_bf16x2(__uint_as_float(r[8 * u + 6]) * inv_l,
                                      __uint_as_float(r[8 * u + 7]) * inv_l);
                    const int chunk = ((c & 1) * 4 + u) ^ (row & 7);
                    *reinterpret_cast<uint4*>(stage + box * C::BOX_BYTES + row * 128 +
                                              chunk * 16) = w;
                }
            }
            fence_async_smem();
        }
        named_bar_sync(5, 256);
        if (ok && threadIdx.x == 64 && !*abort_flag) {
            for (int kb = 0; kb < C::KB; ++kb)
                tma_store_3d(&tm_o, s_q + kb * C::BOX_BYTES, kb * 64, qt * C::BM, bh);
            bulk_commit();
            bulk_wait_read_all();  // the Q buffer stays in place until read
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
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = fwd_bf16_kernel<D, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.N + C::BM - 1) / C::BM;
    // Enough heads per group that a group fills about one wave of CTAs.
    int group = 128 / n_tiles;
    if (group < 1) group = 1;
    dim3 grid(n_tiles, a.H, a.B);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_o, a.lse,
                                                       a.N, a.B * a.H, n_tiles, group,
                                                       a.scale_log2, a.status, a.timeout_ns);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream) {
    if (a.d == 64) return a.causal ? launch_fwd_t<64, true>(a, stream)
                                   : launch_fwd_t<64, false>(a, stream);
    return a.causal ? launch_fwd_t<128, true>(a, stream) : launch_fwd_t<128, false>(a, stream);
}

}  // namespace fa
