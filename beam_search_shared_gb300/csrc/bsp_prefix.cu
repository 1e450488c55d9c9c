// Prompt (prefix) attention of the cascade on 5th-generation tensor cores
// (TensorRT-LLM PR #21738, "Add opt-in cascade attention for wide beam search
// on KVCM V2", description, the prefix half of the cascade: a request's shared
// prompt is attended a single time for all of its beams; all beam_width x
// GQA-group query rows of a request share one K/V stream, which makes Q*K^T and
// P*V dense contractions).
//
// Work unit = (request b, kv head g, query-row block, key range of the plan's
// 64-key tiles). Query rows of a block are (beam w, head j) pairs,
// row = w_local * G + j, at most 128 (the MMA M). Only the valid prompt rows
// [0, P_b) are read (TensorRT-Model-Connect PR #2202, "prefill and decode over
// the cached prefix, not the whole KV allocation"). The kernel walks a unit's
// key range in tiles of TK keys (128 at head_dim <= 128, 64 at 256); the last
// tile of a unit may be partial.
//
// Persistent: one CTA per SM walks its own list of units (the host deals them
// so that the largest per-CTA load is small). Every ring is indexed by a tile
// counter that runs across units, so the producer prefetches the next unit's
// Q and K/V while the current one is still being reduced, and the output of a
// finished unit is written by warps of its own while the next unit's tiles go
// through the tensor core and the softmax.
//
// Warp roles (320 threads):
//   warp 0     TMA producer: Q of each unit into one of NQ shared-memory
//              buffers (3-D box [W_blk][G][64]) and the K and V of the unit's
//              pages (beam 0's prompt pages) into a KST-deep K ring and a
//              VST-deep V ring, one 2-D box of min(page, 64) rows x 64 columns
//              per page slice, column half and tensor, each lane issuing its
//              own boxes; a tile's column half c of K (or V) is a
//              128-byte-swizzled region of TK rows; page ids come from a
//              32-entry window held one per lane. A K slot is released as soon
//              as Q*K^T has read it, a V slot after P*V, Q after the unit's
//              last Q*K^T;
//   warp 1     TMEM allocation; one thread issues tcgen05.mma:
//              S[t%2] = Q K_t^T (both operands in shared memory), then
//              O[k%NO] (+)= P_{t-1} V_{t-1} (unit k);
//   warps 2-5  softmax: thread <-> query row <-> TMEM lane; reads S from TMEM
//              in 32-column chunks twice (row maximum, then probabilities),
//              masks keys >= P_b, online softmax in base 2 with a lazy rescale
//              of O (only when a row maximum grows by more than 2^8), writes P
//              (16-bit pairs) over the first TK/2 columns of its own S buffer,
//              where P*V reads it as the A operand, zeroes V rows past the
//              valid keys of a unit's last tile, and hands each row's running
//              maximum and sum to the epilogue warps at the end of a unit;
//   warps 6-9  epilogue: once a unit's last P*V is done, write the normalised
//              fp32 partial O and its log2-sum-exp2, then release that O
//              buffer. For a request the plan marks fused (its prompt is one
//              key range and each row block's beams hold at most 4 * TK tail
//              keys together) the unit ends with up to four tail tiles (the
//              block's tail keys, beam-major): the epilogue warps resolve each
//              tail key through cache_indirection and the beam's page table,
//              copy its K and V rows into the ring slots the producer hands
//              over (by a counter; 16-byte cp.async into the swizzled layout a
//              TMA box would have; absent keys are zero rows), and publish
//              which keys are readable (one byte per key column and tile); the
//              softmax keeps only a row's own beam's keys of a tail tile. Such
//              a unit writes the final O (q dtype) and LSE of its rows, and the
//              tail kernel skips the request.
// TMEM columns: S0 [0,TK), S1 [TK,2TK) (P_t aliases the first TK/2 columns of
// S[t%2]: tcgen05.mma instructions issued by one thread execute in issue
// order, and the Q*K^T that overwrites S[t%2] is issued after the P*V that
// reads P_t), then NO O buffers of D columns (two where they fit, one at
// head_dim 256).
// Every wait is bounded (1 s without progress); on expiry the CTA flags
// BSP_DEVFLAG_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "bsp_internal.h"
#include "bsp_prompt.cuh"
#include "bsp_ptx.cuh"
#include "../../include/bsp.h"

namespace bsp {

// SPLIT: the half-row layout, whose MMAs have M = 64 (the accumulator's 64 rows sit in TMEM
// lanes 0-15 of each quadrant), so a Q buffer holds 64 rows and the K ring gets a third slot
template <int D, bool SPLIT>
struct PrefixCfg {
    static constexpr int TK = D <= 128 ? 128 : 64;            // keys per tile
    static constexpr int NC = D / 64;                        // 128-byte column regions per row
    static constexpr int NQ = D <= 128 ? 2 : 1;              // Q buffers
    static constexpr int MR = SPLIT ? 64 : kRowsPerBlock;    // MMA M: query rows of a Q buffer
    static constexpr int KST = D == 64 ? (SPLIT ? 6 : 4) : (SPLIT ? 3 : 2);  // K ring depth
    static constexpr int VST = D == 64 ? 7 : 3;              // V ring depth
    static constexpr int Q_BYTES = MR * D * 2;               // NC regions of MR rows x 128 B
    static constexpr int KV_BYTES = TK * D * 2;              // one K (or V) tile
    static constexpr int OFF_K = NQ * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
    static constexpr int OFF_STATS = OFF_V + VST * KV_BYTES;  // float m[128], l[128]
    static constexpr int OFF_TROW = OFF_STATS + 2 * kRowsPerBlock * 4;  // int pool row of tail key c [TK]
    static constexpr int OFF_BAR = OFF_TROW + TK * 4;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;        // barriers + alignment slack
    static constexpr int S_COL = 0;                          // S[0], S[1]: TK fp32 columns each
    static constexpr int O_COL = 2 * TK;                     // O[0] (, O[1]): D fp32 columns each
    static constexpr int NO = (O_COL + 2 * D <= 512) ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(O_COL + NO * D <= 512, "tensor memory");
    static_assert(TK % 64 == 0 && TK / 16 <= 8 && D / 16 <= 16, "tile shape");
    static_assert(TK == prefix_tile_keys(D), "the host's fused-tail bound");
    static constexpr int TAIL_CHUNKS = TK * (D / 8) / 128;  // 16-byte chunks per epilogue thread and tensor
    static constexpr int THREADS = 320;
};

struct PrefixBarriers {
    uint64_t k_full[8];
    uint64_t k_empty[8];  // KST <= 8; arrived by softmax warp 2 when it sees the tile's S complete
    uint64_t v_full[8];
    uint64_t v_empty[8];  // VST <= 8; the tile's P*V completed (also what a rescale of O waits for)
    uint64_t q_full[2];   // Q of unit k landed in shared-memory buffer k % NQ
    uint64_t q_empty[2];  // ... and its last Q*K^T completed
    uint64_t s_full[2];
    uint64_t p_full[2];   // tile t arrives on p_full[t % 2]
    uint64_t o_final[2];  // the last P*V of unit k completes o_final[k % 2]
    uint64_t o_free[2];   // the epilogue of unit k has read O[k % NO]
    uint64_t st_full;     // row statistics of a unit written
    uint64_t st_empty;    // ... and read by the epilogue warps
    uint64_t fill_done[2];  // tail tile n: each epilogue warp has stored its part of it
    uint64_t tail_ready[8]; // tail tile n complete, with its key-validity words: barrier n % 8 (the epilogue
                            // warps run at most KST < 8 tail tiles ahead of the softmax)
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int tail_granted;  // tail tiles whose ring slots the producer has handed to the epilogue warps
};

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s without progress
constexpr uint64_t kDrainNs = 200000000ull;

// a fused unit with tail positions ends with ceil(W_blk * T / TK) (at most kPrefixMaxTailTiles) tiles of
// its beams' tail keys, beam-major: key column c = w_local * T + t of the unit's tail key list
template <int TK>
__device__ __forceinline__ int tail_tiles(const UnitInfo& ui, int wblk) {
    if (!(ui.fused && ui.T > 0)) return 0;
    return (min(wblk, ui.rows - ui.rb * wblk) * ui.T + TK - 1) / TK;
}
template <int TK>
__device__ __forceinline__ int unit_tiles(const UnitInfo& ui, int wblk) {
    return prompt_tiles<TK>(ui) + tail_tiles<TK>(ui, wblk);
}

template <int D, bool BF16, bool SPLIT>
__global__ void __launch_bounds__(320, 1)
prefix_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefixParams p) {
    using C = PrefixCfg<D, SPLIT>;
    constexpr int TK = C::TK, NC = C::NC, NQ = C::NQ, KST = C::KST, VST = C::VST, NO = C::NO, MR = C::MR;
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(!SPLIT || TK == 128, "half-row softmax: 128-key tiles");
    static_assert(KST < 8, "tail_ready: the epilogue warps run at most KST tail tiles ahead of the softmax");
    // Score, probability and output columns a thread handles: all of its row's (dense), or half of
    // them with two threads per row (SPLIT: query rows in TMEM lanes 0-15 of each quadrant, threads
    // t and t + 16 of a warp on the same row through the 16x32bx2 access shape)
    constexpr int HC = SPLIT ? TK / 2 : TK;
    constexpr int HD = SPLIT ? D / 2 : D;
    auto ld_s = [](uint32_t a, uint32_t(&r)[32]) {
        if constexpr (SPLIT) tmem_ld16x2_32<TK / 2>(a, r); else tmem_ld32(a, r);
    };
    auto st_p = [](uint32_t a, const uint32_t(&r)[32]) {
        if constexpr (SPLIT) tmem_st16x2_32<TK / 4>(a, r); else tmem_st32(a, r);
    };
    auto ld_o = [](uint32_t a, uint32_t(&r)[32]) {
        if constexpr (SPLIT) tmem_ld16x2_32<D / 2>(a, r); else tmem_ld32(a, r);
    };
    auto st_o = [](uint32_t a, const uint32_t(&r)[32]) {
        if constexpr (SPLIT) tmem_st16x2_32<D / 2>(a, r); else tmem_st32(a, r);
    };
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto q_buf = [&](int k) -> uint8_t* { return smem + (k % NQ) * C::Q_BYTES; };
    auto k_tile = [&](int gt) -> uint8_t* { return smem + C::OFF_K + (gt % KST) * C::KV_BYTES; };
    auto v_tile = [&](int gt) -> uint8_t* { return smem + C::OFF_V + (gt % VST) * C::KV_BYTES; };
    float* st_m = reinterpret_cast<float*>(smem + C::OFF_STATS);  // [128]
    float* st_l = st_m + kRowsPerBlock;                            // [128]
    // [kPrefixMaxTailTiles][TK]: per tail tile of the current unit and key column, 1 if the key is readable
    uint8_t* s_tok = smem + C::OFF_TROW;
    static_assert(kPrefixMaxTailTiles * TK <= TK * 4, "tail-key flags fit the table area");
    PrefixBarriers* bars = reinterpret_cast<PrefixBarriers*>(smem + C::OFF_BAR);
    volatile int* abort_flag = &bars->abort_flag;

    if (p.graph_hdr != nullptr) {
        // a launch replayed from a CUDA graph: the plan staged since must have the captured shape
        const int4 h0 = __ldg(reinterpret_cast<const int4*>(p.graph_hdr));
        const int4 h1 = __ldg(reinterpret_cast<const int4*>(p.graph_hdr) + 1);
        if (h0.z != p.graph_batch || h1.x != p.W || h1.y != static_cast<int>(gridDim.x) || h1.z != 0) {
            if (threadIdx.x == 0) atomicOr(p.status, BSP_DEVFLAG_GRAPH);
            return;
        }
    }
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int u_begin = __ldg(p.cta_off + blockIdx.x);
    const int u_end = __ldg(p.cta_off + blockIdx.x + 1);
    const int nunits = u_end - u_begin;
    const int ps = 1 << p.ps_log2;

    // ---- setup
    if (tid == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->q_full[i], 1);
            mbar_init(&bars->q_empty[i], 1);  // the MMA thread, after the unit's last Q*K^T
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->p_full[i], 4);   // one arrival per softmax warp
            mbar_init(&bars->o_final[i], 1);
            mbar_init(&bars->o_free[i], 4);   // one arrival per epilogue warp
        }
        mbar_init(&bars->st_full, 4);   // one arrival per softmax warp
        mbar_init(&bars->st_empty, 4);  // one arrival per epilogue warp
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->fill_done[i], 4);  // one arrival per epilogue warp
        }
        for (int i = 0; i < 8; ++i) mbar_init(&bars->tail_ready[i], 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        bars->tail_granted = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 1) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
    // zero the query rows no TMA box covers, so padded rows stay finite: rows past W_blk * G, or
    // (SPLIT) the rows of each 16-row quadrant block past its bq * G
    {
        constexpr int NCHUNK = NQ * NC * MR * 8;  // 16-byte chunks of the Q buffers
        for (int idx = tid; idx < NCHUNK; idx += C::THREADS) {
            const int r = (idx >> 3) % MR;
            const bool covered = SPLIT ? (r & 15) < p.bq * p.G : r < p.Wblk * p.G;
            if (!covered) reinterpret_cast<uint4*>(smem)[idx] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // every CTA of this grid is resident: a dependent launch (the tail kernel) may start on the
    // SMs this grid leaves; it waits for this grid's completion before reading the partials
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ================= TMA producer =================
        const int BR = ps < kTileKeys ? ps : kTileKeys;  // rows per box (a page, or 64 rows of a larger page)
        int gt = 0, k = 0, ntail = 0;
        bool ok = true;
        for (int u = u_begin; u < u_end && ok; ++u, ++k) {
            const UnitInfo ui = load_unit(p, u);
            const int qb = k % NQ;
            if (k >= NQ) {
                ok = mbar_wait(&bars->q_empty[qb], ((k / NQ) - 1) & 1, abort_flag, kWaitTimeoutNs);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
            }
            if (lane == 0) {
                if constexpr (SPLIT) {
                    // M rows 16i .. 16i + bq*G - 1 (TMEM lanes 32i ..): beams i*bq .. of the block (box
                    // [bq][G][64])
                    mbar_arrive_expect_tx(&bars->q_full[qb], NC * 4 * p.bq * p.G * 128);
                    for (int c = 0; c < NC; ++c)
                        for (int i = 0; i < 4; ++i)
                            tma_load_3d(q_buf(k) + c * MR * 128 + i * 16 * 128, &tm_q, &bars->q_full[qb],
                                        c * 64, ui.g * p.G, ui.row_off + ui.rb * p.Wblk + i * p.bq);
                } else {
                    mbar_arrive_expect_tx(&bars->q_full[qb], NC * p.Wblk * p.G * 128);
                    for (int c = 0; c < NC; ++c)
                        tma_load_3d(q_buf(k) + c * MR * 128, &tm_q, &bars->q_full[qb], c * 64,
                                    ui.g * p.G, ui.row_off + ui.rb * p.Wblk);
                }
            }
            const int ntiles = unit_tiles<TK>(ui, p.Wblk);
            const int ptiles = prompt_tiles<TK>(ui);
            const int* pg = p.pages + ui.page_off;
            const int npages = (ui.P + ps - 1) >> p.ps_log2;
            int win_base = -1, my_page = 0;
            for (int t = 0; t < ntiles; ++t, ++gt) {
                if (gt >= KST) {
                    ok = mbar_wait(&bars->k_empty[gt % KST], ((gt / KST) - 1) & 1, abort_flag, kWaitTimeoutNs);
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                }
                if (t >= ptiles) {
                    // a tail tile: the epilogue warps gather it once both slots are free
                    if (gt >= VST) {
                        ok = mbar_wait(&bars->v_empty[gt % VST], ((gt / VST) - 1) & 1, abort_flag, kWaitTimeoutNs);
                        ok = __all_sync(FULL, ok);
                        if (!ok) break;
                    }
                    // hand them over by a counter: the producer may run several tail tiles ahead of the
                    // epilogue warps (short units, deep rings), which a parity wait could not follow
                    ++ntail;
                    if (lane == 0) counter_release(&bars->tail_granted, ntail);
                    __syncwarp();
                    continue;
                }
                const int key0 = ui.key_begin + t * TK;
                const int valid = min(TK, ui.key_end - key0);
                const int nchunks = (valid + BR - 1) / BR;  // pages (or 64-row slices) with valid keys
                const int tile_bytes = nchunks * BR * D * 2;
                const int pidx0 = key0 >> p.ps_log2;
                const int pidx_last = (key0 + (nchunks - 1) * BR) >> p.ps_log2;
                if (win_base < 0 || pidx_last >= win_base + 32) {  // warp-uniform
                    win_base = pidx0;
                    my_page = (win_base + lane < npages) ? __ldg(pg + win_base + lane) : 0;
                }
                // box b of a tensor: column half b % NC of chunk b / NC
                const int nbox = nchunks * NC;
                for (int tensor = 0; tensor < 2; ++tensor) {
                    if (tensor == 1 && gt >= VST) {
                        ok = mbar_wait(&bars->v_empty[gt % VST], ((gt / VST) - 1) & 1, abort_flag, kWaitTimeoutNs);
                        ok = __all_sync(FULL, ok);
                        if (!ok) break;
                    }
                    uint64_t* full = tensor == 0 ? &bars->k_full[gt % KST] : &bars->v_full[gt % VST];
                    uint8_t* base = tensor == 0 ? k_tile(gt) : v_tile(gt);
                    const CUtensorMap* map = tensor == 0 ? &tm_k : &tm_v;
                    if (lane == 0) mbar_arrive_expect_tx(full, tile_bytes);
                    for (int b0 = 0; b0 < nbox; b0 += 32) {
                        const int bx = b0 + lane;
                        const int ch = min(bx / NC, nchunks - 1);
                        const int key = key0 + ch * BR;
                        int page = __shfl_sync(FULL, my_page, (key >> p.ps_log2) - win_base);
                        if (bx < nbox) {
                            if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
                                atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
                                page = 0;
                            }
                            const int c = bx % NC;
                            const int row = ((page * p.Hkv + ui.g) << p.ps_log2) + (key & (ps - 1));
                            tma_load_2d(base + c * TK * 128 + ch * BR * 128, map, full, c * 64, row);
                        }
                    }
                }
                if (!ok) break;
                __syncwarp();
            }
        }
        if (!ok) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
            }
            // drain: let this CTA's own copies land before the CTA exits
            const uint64_t t0 = globaltimer_ns();
            for (int j = max(0, gt - KST); j <= gt; ++j)
                while (!mbar_try_wait(&bars->k_full[j % KST], (j / KST) & 1) && globaltimer_ns() - t0 < kDrainNs) {
                }
            for (int j = max(0, gt - VST); j <= gt; ++j)
                while (!mbar_try_wait(&bars->v_full[j % VST], (j / VST) & 1) && globaltimer_ns() - t0 < kDrainNs) {
                }
            for (int j = max(0, k - NQ); j <= k; ++j)
                while (!mbar_try_wait(&bars->q_full[j % NQ], (j / NQ) & 1) && globaltimer_ns() - t0 < kDrainNs) {
                }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t ID_QK = idesc_f16(MR, TK, BF16, false);
            constexpr uint32_t ID_PV = idesc_f16(MR, D, BF16, true);
            int gt = 0, k = 0;
            int pend = -1, pend_unit = 0;  // tile whose P*V is not issued yet, and its unit
            bool pend_first = false, pend_last = false;
            bool ok = true;
            // (V first: its load does not depend on the softmax, and a wait that has already completed
            // still costs a shared-memory round trip, which would otherwise sit between P and the MMAs)
            auto issue_pv = [&](int j, int unit, bool first, bool last) -> bool {
                if (!mbar_wait(&bars->v_full[j % VST], (j / VST) & 1, abort_flag, kWaitTimeoutNs)) return false;
                if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, abort_flag, kWaitTimeoutNs)) return false;
                if (first && unit >= NO) {
                    // O[unit % NO] was last used by unit - NO: its epilogue must have read it
                    const int f = unit - NO;
                    if (!mbar_wait(&bars->o_free[f & 1], (f >> 1) & 1, abort_flag, kWaitTimeoutNs)) return false;
                }
                tc_fence_after();
                const uint32_t p_tmem = tmem + C::S_COL + (j & 1) * TK;
                const uint32_t o_tmem = tmem + C::O_COL + (unit % NO) * D;
                const uint32_t v_addr = smem_u32(v_tile(j));
#pragma unroll
                for (int kk = 0; kk < TK / 16; ++kk) {
                    const uint64_t bd = sdesc_sw128(v_addr + kk * 16 * 128, TK * 128, 1024);
                    mma_f16_tmem_a(o_tmem, p_tmem + kk * 8, bd, ID_PV, (!first || kk > 0) ? 1u : 0u);
                }
                // one commit per batch of MMAs: a commit right after another holds this thread until the
                // first one's MMAs finish. v_empty also tells the softmax that this P*V is done (its
                // rescale of O), and the K slot is handed back by a softmax warp (s_full)
                mma_commit(&bars->v_empty[j % VST]);
                if (last) mma_commit(&bars->o_final[unit & 1]);
                return true;
            };
            for (int u = u_begin; u < u_end && ok; ++u, ++k) {
                const int ntiles = unit_tiles<TK>(load_unit(p, u), p.Wblk);
                const int qb = k % NQ;
                ok = mbar_wait(&bars->q_full[qb], (k / NQ) & 1, abort_flag, kWaitTimeoutNs);
                if (!ok) break;
                const uint32_t q_addr = smem_u32(q_buf(k));
                for (int t = 0; t < ntiles; ++t, ++gt) {
                    ok = mbar_wait(&bars->k_full[gt % KST], (gt / KST) & 1, abort_flag, kWaitTimeoutNs);
                    if (!ok) break;
                    // S[gt % 2] holds P of tile gt - 2, whose P*V was issued before this Q*K^T
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(k_tile(gt));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t ad =
                            sdesc_sw128(q_addr + (kk >> 2) * (MR * 128) + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(k_addr + (kk >> 2) * (TK * 128) + (kk & 3) * 32, 16, 1024);
                        mma_f16(tmem + C::S_COL + (gt & 1) * TK, ad, bd, ID_QK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars->s_full[gt & 1]);
                    if (t == ntiles - 1) mma_commit(&bars->q_empty[qb]);  // Q no longer read
                    if (pend >= 0) {
                        ok = issue_pv(pend, pend_unit, pend_first, pend_last);
                        if (!ok) break;
                    }
                    pend = gt;
                    pend_unit = k;
                    pend_first = t == 0;
                    pend_last = t == ntiles - 1;
                }
            }
            if (ok && pend >= 0) ok = issue_pv(pend, pend_unit, pend_first, pend_last);
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
            }
            // drain: every MMA issued by this thread completes before TMEM is freed
            mma_commit(&bars->drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&bars->drain, 0) && globaltimer_ns() - t0 < kDrainNs) {
            }
        }
    } else if (warp < 6) {
        // ================= softmax warps =================
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int half = SPLIT ? lane >> 4 : 0;                 // which half of the row's columns
        const int row = quad * 32 + (SPLIT ? (lane & 15) : lane);  // TMEM lane of the thread's query row
        // beam (within the row block) of the row
        const int beam = SPLIT ? quad * p.bq + (lane & 15) / p.G : row / p.G;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float sl2 = p.scale_log2;
        bool ok = true;
        int gt = 0, ntail = 0;
        for (int k = 0; k < nunits && ok; ++k) {
            const UnitInfo cur = load_unit(p, u_begin + k);
            const int ntiles = unit_tiles<TK>(cur, p.Wblk);
            const int ptiles = prompt_tiles<TK>(cur);
            const int nw = min(p.Wblk, cur.rows - cur.rb * p.Wblk);  // beams (prompt tokens) of the block
            // the row's own beam's keys in the unit's tail key list: columns [lo, lo + T)
            const int lo = beam * cur.T, hi = lo + cur.T;
            const uint32_t o_col = C::O_COL + (k % NO) * D;
            // a warp whose 32 rows are all padding skips the arithmetic but keeps the
            // barrier protocol (the p_full ordering below keeps its arrivals in the right phase)
            const bool warp_live = SPLIT ? quad * p.bq < nw : quad * 32 < nw * p.G;
            float m = -INFINITY, l = 0.f;
            for (int t = 0; t < ntiles; ++t, ++gt) {
                const bool tail = t >= ptiles;  // a tail tile (zero-filled past its keys)
                const int tn = t - ptiles;      // its index among the unit's tail tiles
                const int valid = tail ? TK : min(TK, cur.key_end - (cur.key_begin + t * TK));
                ok = mbar_wait(&bars->s_full[gt & 1], (gt >> 1) & 1, abort_flag, kWaitTimeoutNs);
                // S complete: this tile's Q*K^T has read its K slot; one thread hands it back
                if (ok && warp == 2 && lane == 0) mbar_arrive(&bars->k_empty[gt % KST]);
                if (ok && tail) {
                    // the tail tile's key-validity words. The epilogue warps gather tail tile n only once the
                    // producer has the slot of the tile KST positions earlier back, which needs this
                    // warp's S wait for that tile: they run at most KST < 8 tail tiles ahead, so a parity
                    // wait on barrier n % 8 names the right phase.
                    ok = mbar_wait(&bars->tail_ready[ntail & 7], (ntail >> 3) & 1, abort_flag, kWaitTimeoutNs);
                    ++ntail;
                }
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc_fence_after();
                if (warp_live) {
                    const uint32_t s_col = lane_base + C::S_COL + (gt & 1) * TK;
                    // masked keys count as -inf: they take no part in the maximum and their probability
                    // exp2(-inf) is 0. A prompt tile masks keys >= P_b (a unit's partial last tile only),
                    // the tail tile every key but the row's own beam's readable ones.
                    // a causal prefill row t sees keys 0 .. C + t: its own count of valid keys in this tile
                    int rvalid = valid;
                    if (cur.causal >= 0)
                        rvalid = min(valid, cur.causal + cur.rb * p.Wblk + beam + 1 - (cur.key_begin + t * TK));
                    const bool partial = valid < TK || tail || (cur.causal >= 0 && __any_sync(FULL, rvalid < TK));
                    const uint32_t ninf = __float_as_uint(-INFINITY);
                    // kept columns of a partial tile, one bit per key: [0, valid) of a prompt tile; of the
                    // tail tile the row's own beam's columns [lo, lo + T) (T <= 8, so they span at most two
                    // 32-bit words) whose key is readable
                    uint32_t km[TK / 32];
                    if (partial) {
                        uint64_t win = 0;
                        // the row's columns in this tail tile, [c0, c1)
                        const int c0 = max(lo - tn * TK, 0), c1 = min(hi - tn * TK, TK);
                        const int wbase = c0 & ~31;
                        if (tail)
                            for (int c = c0; c < c1; ++c)
                                if (s_tok[tn * TK + c]) win |= 1ull << (c - wbase);
#pragma unroll
                        for (int j = 0; j < TK / 32; ++j) {
                            const int n = min(max(rvalid - 32 * j, 0), 32);
                            const uint32_t pm = n == 32 ? ~0u : (1u << n) - 1u;
                            const uint32_t tm = 32 * j == wbase        ? static_cast<uint32_t>(win)
                                                : 32 * j == wbase + 32 ? static_cast<uint32_t>(win >> 32)
                                                                       : 0u;
                            km[j] = tail ? tm : pm;
                        }
                    }
                    // the two mask words of tile columns [c0, c0 + 64) (c0 is 0 or 64)
                    auto mask_pair = [&](int c0, uint32_t& ma, uint32_t& mb) {
                        ma = km[0];
                        mb = km[1];
                        if constexpr (TK > 64) {
                            if (c0 != 0) {
                                ma = km[2];
                                mb = km[3];
                            }
                        }
                    };
                    // pass 1: the row maximum of the raw scores, then scaled (the scale is positive)
                    float mp[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) mp[j] = -INFINITY;
#pragma unroll 1
                    for (int c0 = 0; c0 < HC; c0 += 64) {
                        uint32_t ma = ~0u, mb = ~0u;
                        if (partial) {
                            mask_pair(c0 + half * HC, ma, mb);
                            if (!__any_sync(FULL, (ma | mb) != 0u)) continue;  // no row of the warp keeps one
                        }
                        uint32_t sa[32], sb[32];
                        ld_s(s_col + c0, sa);
                        ld_s(s_col + c0 + 32, sb);
                        tmem_wait_ld();
                        if (partial && __any_sync(FULL, (ma & mb) != ~0u)) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                sa[c] = (ma >> c) & 1u ? sa[c] : ninf;
                                sb[c] = (mb >> c) & 1u ? sb[c] : ninf;
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            mp[c & 7] = fmaxf(mp[c & 7], __uint_as_float(sa[c]));
                            mp[c & 7] = fmaxf(mp[c & 7], __uint_as_float(sb[c]));
                        }
                    }
                    float mxr = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                      fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
                    if constexpr (SPLIT) mxr = fmaxf(mxr, __shfl_xor_sync(FULL, mxr, 16));  // the row's other half
                    const float mx = mxr * sl2;
                    // lazy maximum: keep the old one unless the row maximum grew by more than 2^8
                    const bool need = t > 0 && mx > m + 8.0f;
                    const bool rescale = __any_sync(FULL, need);
                    float alpha = 1.0f;
                    if (t == 0) {
                        m = mx;
                    } else if (need) {
                        alpha = exp2f(m - mx);
                        m = mx;
                        l *= alpha;
                    }
                    if (rescale) {
                        // O is rescaled only after P*V of the previous tile has finished (the release of
                        // its V slot); P*V of this tile waits for p_full. (The slot's next phase needs
                        // the P*V of tile gt - 1 + VST > gt, whose P this warp has not written yet, so
                        // the phase waited for is exact.)
                        ok = mbar_wait(&bars->v_empty[(gt - 1) % VST], ((gt - 1) / VST) & 1, abort_flag, kWaitTimeoutNs);
                        ok = __all_sync(FULL, ok);
                        if (ok) {
                            tc_fence_after();
#pragma unroll 1
                            for (int c0 = 0; c0 < HD; c0 += 32) {
                                uint32_t orr[32];
                                ld_o(lane_base + o_col + c0, orr);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                                st_o(lane_base + o_col + c0, orr);
                            }
                        }
                    }
                    // pass 2: probabilities 2^(s * scale_log2 - m) and their sum; P in 16-bit pairs
                    // over the first TK/2 columns of this S buffer, 64 keys per store. P columns
                    // [32i, 32i+32) overwrite score columns already read in this pass.
                    const float nm = -m;
                    float rsp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                    for (int c0 = 0; c0 < HC; c0 += 64) {
                        uint32_t ma = ~0u, mb = ~0u;
                        if (partial) mask_pair(c0 + half * HC, ma, mb);
                        uint32_t pk[32];
                        if (partial && !__any_sync(FULL, (ma | mb) != 0u)) {
                            // every key of these 64 columns is masked for the warp's rows: P = 0
#pragma unroll
                            for (int c = 0; c < 32; ++c) pk[c] = 0u;
                            st_p(s_col + (c0 >> 1), pk);
                            continue;
                        }
                        uint32_t sa[32], sb[32];
                        ld_s(s_col + c0, sa);
                        ld_s(s_col + c0 + 32, sb);
                        tmem_wait_ld();
                        if (partial && __any_sync(FULL, (ma & mb) != ~0u)) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                sa[c] = (ma >> c) & 1u ? sa[c] : ninf;
                                sb[c] = (mb >> c) & 1u ? sb[c] : ninf;
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const float p0 = exp2f(fmaf(__uint_as_float(sa[c]), sl2, nm));
                            const float p1 = exp2f(fmaf(__uint_as_float(sa[c + 1]), sl2, nm));
                            const float p2 = exp2f(fmaf(__uint_as_float(sb[c]), sl2, nm));
                            const float p3 = exp2f(fmaf(__uint_as_float(sb[c + 1]), sl2, nm));
                            rsp[(c >> 1) & 1] += p0 + p1;
                            rsp[2 + ((c >> 1) & 1)] += p2 + p3;
                            pk[c >> 1] = pack2<BF16>(p0, p1);
                            pk[16 + (c >> 1)] = pack2<BF16>(p2, p3);
                        }
                        st_p(s_col + (c0 >> 1), pk);
                    }
                    tmem_wait_st();
                    l += (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
                }
                if (!ok) break;
                if (valid < TK) {
                    // a unit's last tile: zero V rows past the valid keys (stale or garbage rows
                    // times P = 0 must not produce NaN)
                    ok = mbar_wait(&bars->v_full[gt % VST], (gt / VST) & 1, abort_flag, kWaitTimeoutNs);
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                    uint8_t* sV = v_tile(gt);
                    const int nzc = (TK - valid) * 8;  // 16-byte chunks per column half
                    for (int c = 0; c < NC; ++c)
                        for (int idx = tid - 64; idx < nzc; idx += 128)
                            reinterpret_cast<uint4*>(sV + c * TK * 128 + valid * 128)[idx] = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                // a warp arrives for this tile only once every warp has arrived for the previous
                // one, so no warp's arrival can land in an earlier tile's phase
                if (gt > 0) {
                    ok = mbar_wait(&bars->p_full[(gt - 1) & 1], ((gt - 1) >> 1) & 1, abort_flag, kWaitTimeoutNs);
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[gt & 1]);
            }
            if (!ok) break;
            // hand the row statistics of this unit to the epilogue warps (they read the
            // previous unit's early in this one)
            if (k >= 1) {
                ok = mbar_wait(&bars->st_empty, (k - 1) & 1, abort_flag, kWaitTimeoutNs);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
            }
            if constexpr (SPLIT) l += __shfl_xor_sync(FULL, l, 16);  // the row's other half
            if (half == 0) {
                st_m[row] = m;
                st_l[row] = l;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->st_full);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
        }
    } else {
        // ================= epilogue warps =================
        constexpr int CH = D / 8;               // 16-byte chunks of a K or V row
        constexpr int RPW = 32 / CH;            // tail-tile rows a warp covers per gather step
        constexpr int RS = kRowsPerBlock / CH;  // row step between one thread's gather steps
        const int quad = warp & 3;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        // tail-tile gather: thread (quad, lane) copies chunk kc = lane % CH of rows
        // quad*RPW + lane/CH + i*RS (i < TAIL_CHUNKS); each lane resolves the pool row of one of the
        // warp's rows (lrow), and the thread copying row quad*RPW + lane/CH + i*RS takes it from lane
        // i*RPW + lane/CH
        const int kc = lane % CH;
        const int lrow = quad * RPW + lane % RPW + (lane / RPW) * RS;
        const bool lrow_ok = lane / RPW < C::TAIL_CHUNKS;
        // pool row of the tail key in column n * TK + lrow of unit ui's tail key list (column c = w_local * T +
        // t is position P_b + t of beam w0 + w_local, read through cache_indirection); -1 past the unit's
        // keys or when the source beam or its page is out of range
        auto tail_row = [&](const UnitInfo& ui, int n) -> int {
            const int w0 = ui.rb * p.Wblk;
            const int nkeys = min(p.Wblk, p.W - w0) * ui.T;
            const int cc = n * TK + lrow;
            if (!lrow_ok || cc >= nkeys) return -1;
            const int wl = cc / ui.T, t = cc - wl * ui.T;
            const int pos = ui.P + t;
            const int src = __ldg(p.ci + (static_cast<long long>(ui.b) * p.W + w0 + wl) * p.max_seq + pos);
            int r = -1;
            if (static_cast<unsigned>(src) < static_cast<unsigned>(p.W)) {
                const int page = __ldg(p.beam_pages + (static_cast<long long>(ui.b) * p.W + src) * p.beam_pages_stride +
                                       (pos >> p.ps_log2));
                if (static_cast<unsigned>(page) < static_cast<unsigned>(p.num_pages))
                    r = ((page * p.Hkv + ui.g) << p.ps_log2) + (pos & (ps - 1));
            }
            if (r < 0) {
                atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
            } else {
                // the gather runs a few tiles later: bring the row's K and V into L2 now
#pragma unroll
                for (int off = 0; off < D * 2; off += 128) {
                    prefetch_l2(static_cast<const uint8_t*>(p.k_pool) + static_cast<long long>(r) * (D * 2) + off);
                    prefetch_l2(static_cast<const uint8_t*>(p.v_pool) + static_cast<long long>(r) * (D * 2) + off);
                }
            }
            return r;
        };
        const uint16_t* k_pool = static_cast<const uint16_t*>(p.k_pool);
        const uint16_t* v_pool = static_cast<const uint16_t*>(p.v_pool);
        bool ok = true;
        int gt = 0, ntail = 0;
        UnitInfo cur;
        int trow[kPrefixMaxTailTiles];  // this lane's resolved tail rows (column n * TK + lrow) of the unit `cur`
        // (loops over the tail tiles are not unrolled, and pick trow[n] by selects: one copy of their
        // code, and trow stays in registers)
        auto pick = [&](int n) -> int { return n == 0 ? trow[0] : n == 1 ? trow[1] : n == 2 ? trow[2] : trow[3]; };
        static_assert(kPrefixMaxTailTiles == 4, "pick");
        auto resolve = [&](const UnitInfo& ui) {
            const int ntt = tail_tiles<TK>(ui, p.Wblk);
#pragma unroll
            for (int n = 0; n < kPrefixMaxTailTiles; ++n) trow[n] = -1;
#pragma unroll 1
            for (int n = 0; n < ntt; ++n) {
                const int r = tail_row(ui, n);
                trow[0] = n == 0 ? r : trow[0];
                trow[1] = n == 1 ? r : trow[1];
                trow[2] = n == 2 ? r : trow[2];
                trow[3] = n == 3 ? r : trow[3];
            }
        };
        if (nunits > 0) {
            cur = load_unit(p, u_begin);
            resolve(cur);
        }
        for (int k = 0; k < nunits && ok; ++k) {
            // gather the unit's tail tiles into the K and V ring slots the producer hands over. The validity
            // words of the unit's tail tiles are free: the softmax finished the previous unit (its
            // statistics were read).
            const int ntt = tail_tiles<TK>(cur, p.Wblk);
#pragma unroll 1
            for (int n = 0; n < ntt; ++n) {
                const int gtt = gt + prompt_tiles<TK>(cur) + n;
                ok = counter_wait(&bars->tail_granted, ntail, abort_flag, kWaitTimeoutNs);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                const int myrow = pick(n);
                if (lrow_ok) s_tok[n * TK + lrow] = myrow >= 0 ? 1 : 0;
                uint8_t* kt = k_tile(gtt);
                uint8_t* vt = v_tile(gtt);
                // (not unrolled: this code runs next to the softmax's, and a smaller instruction footprint
                // keeps the softmax loop in the instruction cache)
#pragma unroll 1
                for (int i = 0; i < C::TAIL_CHUNKS; ++i) {
                    const int r = __shfl_sync(FULL, myrow, i * RPW + lane / CH);
                    const int c = quad * RPW + lane / CH + i * RS;
                    // the layout of a TMA box with 128-byte swizzle: chunk kc of row c in column half kc/8
                    const uint32_t off = (kc >> 3) * (TK * 128) + c * 128 + (((kc & 7) ^ (c & 7)) << 4);
                    const long long e = static_cast<long long>(r < 0 ? 0 : r) * D + kc * 8;
                    const uint32_t nb = r < 0 ? 0u : 16u;  // absent keys are zero rows
                    cp_async16(kt + off, k_pool + e, nb);
                    cp_async16(vt + off, v_pool + e, nb);
                }
                cp_async_commit_wait_all();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->fill_done[ntail & 1]);
                if (quad == 0) {
                    if (lane == 0) {
                        // (each warp arrives for tail tile n + 2 only after arriving for n + 1, so this
                        // warp's own arrival keeps the phase waited for exact)
                        ok = mbar_wait(&bars->fill_done[ntail & 1], (ntail >> 1) & 1, abort_flag, kWaitTimeoutNs);
                        if (ok) {
                            mbar_arrive(&bars->k_full[gtt % KST]);
                            mbar_arrive(&bars->v_full[gtt % VST]);
                            mbar_arrive(&bars->tail_ready[ntail & 7]);
                        }
                    }
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                }
                ++ntail;
            }
            if (!ok) break;
            gt += unit_tiles<TK>(cur, p.Wblk);
            const int w0 = cur.rb * p.Wblk;
            const int nw = min(p.Wblk, cur.rows - w0);
            // the thread's query row: TMEM lane orow, beam wl of the block, head jh of the group; with
            // SPLIT two threads per row, each writing half of its columns
            const int r16 = lane & 15, ohalf = SPLIT ? lane >> 4 : 0;
            const int orow = quad * 32 + (SPLIT ? r16 : lane);
            const int wl = SPLIT ? quad * p.bq + r16 / p.G : orow / p.G;
            const int jh = SPLIT ? r16 % p.G : orow % p.G;
            const bool warp_live = SPLIT ? quad * p.bq < nw : quad * 32 < nw * p.G;
            const bool live = SPLIT ? (r16 < p.bq * p.G && wl < nw) : orow < nw * p.G;
            ok = mbar_wait(&bars->st_full, k & 1, abort_flag, kWaitTimeoutNs);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            const float m = st_m[orow];
            const float l = st_l[orow];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->st_empty);
            // resolve the next unit's tail keys while this unit's last P*V runs
            const UnitInfo done = cur;
            if (k + 1 < nunits) {
                cur = load_unit(p, u_begin + k + 1);
                resolve(cur);
            }
            ok = mbar_wait(&bars->o_final[k & 1], (k >> 1) & 1, abort_flag, kWaitTimeoutNs);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc_fence_after();
            const float inv = 1.0f / l;
            const uint32_t o_col = C::O_COL + (k % NO) * D;
            const int cb = ohalf * HD;  // first output column of the thread
            if (done.fused) {
                // the request's whole key set went through this unit: the final O (q dtype) and LSE
                const long long rh = (static_cast<long long>(done.row_off) + (w0 + wl)) * p.Hq + done.g * p.G + jh;
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + rh * D);
#pragma unroll 1
                for (int c0 = 0; c0 < HD && warp_live; c0 += 32) {
                    uint32_t orr[32];
                    ld_o(lane_base + o_col + c0, orr);
                    tmem_wait_ld();
                    if (live) {
                        uint4 w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float* f = reinterpret_cast<const float*>(orr) + 8 * e;
                            w[e] = make_uint4(pack2<BF16>(f[0] * inv, f[1] * inv), pack2<BF16>(f[2] * inv, f[3] * inv),
                                              pack2<BF16>(f[4] * inv, f[5] * inv), pack2<BF16>(f[6] * inv, f[7] * inv));
                        }
                        // rows and column halves start at multiples of 64 bytes: 32-byte stores when o is
                        // 32-byte aligned
                        if ((reinterpret_cast<uintptr_t>(p.o) & 31u) == 0) {
                            st_global_v8(dst + ((cb + c0) >> 3), w[0], w[1]);
                            st_global_v8(dst + ((cb + c0) >> 3) + 2, w[2], w[3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) dst[((cb + c0) >> 3) + e] = w[e];
                        }
                    }
                }
                if (live && ohalf == 0) {
                    const float lse2 = m + log2f(l);
                    p.lse[rh] = p.lse_base2 ? lse2 : lse2 * 0.69314718055994530942f;
                }
            } else {
                const long long prow =
                    (static_cast<long long>(done.part) * p.W + (w0 + wl)) * p.Hq + done.g * p.G + jh;
                float4* dst = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll 1
                for (int c0 = 0; c0 < HD && warp_live; c0 += 32) {
                    uint32_t orr[32];
                    ld_o(lane_base + o_col + c0, orr);
                    tmem_wait_ld();
                    if (live) {
                        // (the workspace's partial rows are 32-byte aligned)
#pragma unroll
                        for (int e = 0; e < 8; e += 2)
                            st_global_v8(dst + ((cb + c0) >> 2) + e,
                                         make_uint4(__float_as_uint(__uint_as_float(orr[4 * e]) * inv),
                                                    __float_as_uint(__uint_as_float(orr[4 * e + 1]) * inv),
                                                    __float_as_uint(__uint_as_float(orr[4 * e + 2]) * inv),
                                                    __float_as_uint(__uint_as_float(orr[4 * e + 3]) * inv)),
                                         make_uint4(__float_as_uint(__uint_as_float(orr[4 * e + 4]) * inv),
                                                    __float_as_uint(__uint_as_float(orr[4 * e + 5]) * inv),
                                                    __float_as_uint(__uint_as_float(orr[4 * e + 6]) * inv),
                                                    __float_as_uint(__uint_as_float(orr[4 * e + 7]) * inv)));
                    }
                }
                if (live && ohalf == 0) p.part_lse[prow] = m + log2f(l);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free[k & 1]);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool BF16, bool SPLIT>
static cudaError_t prepare_prefix_k() {
    using C = PrefixCfg<D, SPLIT>;
    static_assert(sizeof(PrefixBarriers) <= 512, "barrier block");
    static_assert(C::SMEM <= 227 * 1024, "shared memory");
    cudaError_t e =
        cudaFuncSetAttribute(prefix_attn_kernel<D, BF16, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(prefix_attn_kernel<D, BF16, SPLIT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

// the half-row variant exists for 128-key tiles (head_dim <= 128)
template <int D, bool BF16>
static cudaError_t prepare_prefix_t() {
    cudaError_t e = prepare_prefix_k<D, BF16, false>();
    if constexpr (PrefixCfg<D, true>::TK == 128)
        if (e == cudaSuccess) e = prepare_prefix_k<D, BF16, true>();
    return e;
}

template <int D, bool BF16>
static cudaError_t launch_prefix_t(int ctas, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const PrefixParams& p, cudaStream_t stream) {
    if constexpr (PrefixCfg<D, true>::TK == 128) {
        using CS = PrefixCfg<D, true>;
        if (p.bq > 0) {
            prefix_attn_kernel<D, BF16, true><<<ctas, CS::THREADS, CS::SMEM, stream>>>(tq, tk, tv, p);
            return cudaGetLastError();
        }
    }
    if (p.bq > 0) return cudaErrorInvalidValue;
    using C = PrefixCfg<D, false>;
    prefix_attn_kernel<D, BF16, false><<<ctas, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

cudaError_t prepare_prefix(int head_dim, bool bf16) {
    switch (head_dim) {
        case 64: return bf16 ? prepare_prefix_t<64, true>() : prepare_prefix_t<64, false>();
        case 128: return bf16 ? prepare_prefix_t<128, true>() : prepare_prefix_t<128, false>();
        case 256: return bf16 ? prepare_prefix_t<256, true>() : prepare_prefix_t<256, false>();
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_prefix(int head_dim, bool bf16, int ctas, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const PrefixParams& p, cudaStream_t stream) {
    if (ctas == 0 || p.num_units == 0) return cudaSuccess;
    switch (head_dim) {
        case 64: return bf16 ? launch_prefix_t<64, true>(ctas, tq, tk, tv, p, stream)
                             : launch_prefix_t<64, false>(ctas, tq, tk, tv, p, stream);
        case 128: return bf16 ? launch_prefix_t<128, true>(ctas, tq, tk, tv, p, stream)
                              : launch_prefix_t<128, false>(ctas, tq, tk, tv, p, stream);
        case 256: return bf16 ? launch_prefix_t<256, true>(ctas, tq, tk, tv, p, stream)
                              : launch_prefix_t<256, false>(ctas, tq, tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bsp
