// Prompt (prefix) attention of the cascade for wide beams, on 5th-generation
// tensor cores (TensorRT-LLM PR #21738, "Add opt-in cascade attention for wide
// beam search on KVCM V2", description, Problem and Solution: a request's shared
// prompt is attended a single time for all of its beams; the workload the
// method was built for has batch 128, beam 96 and a ~3k-token prompt).
//
// When a (request b, kv head g) has more query rows W * G than one MMA holds
// (128 < W * G <= 256), splitting them into row blocks that run as separate
// units streams the prompt K/V once per block. Here one CTA holds all of them:
// two M = 128 blocks, X = A (beams [0, Wb)) and X = B (beams [Wb, W)),
// Wb = ceil(W / 2), which share every K/V tile in shared memory. Each block's
// beams are spread over the four TMEM lane quadrants (bq = ceil(Wb / 4) beams,
// bq * G rows, per quadrant; the rest of a quadrant is zero padding), so the
// softmax work of a block is even over the four SM sub-partitions.
//
// Work unit = (request b, kv head g, key range of the plan's 64-key tiles).
// Only the valid prompt rows [0, P_b) are read (TensorRT-Model-Connect PR #2202,
// "prefill and decode over the cached prefix, not the whole KV allocation").
// A unit the plan marks fused (one key range, at most kWideMaxTailTiles tiles of
// tail keys) ends with ceil(W * T_b / 128) tail tiles: the tail keys of all W
// beams, beam-major (key column w * T_b + t is position P_b + t of beam w, read
// through cache_indirection and that beam's page table); every row keeps only
// its own beam's columns. Such a unit writes the final O and LSE (the tail
// attention and the log-sum-exp merge are the same online softmax), other units
// write fp32 partial states for the tail kernel.
//
// A prefill at head_dim <= 128 runs here too: a unit is (request b, kv head g,
// pair of row blocks rb), block X holding prompt tokens [(2 rb + X) Wb,
// (2 rb + X + 1) Wb), Wb = 4 floor(32 / G), and in a causal prefill each row
// masks the keys past its own position (token t sees the C_b cached rows and
// tokens 0 .. t). The pair reads each K/V tile once for up to 256 rows. A
// request whose cached rows the plan cut into key ranges writes one fp32
// partial state per range, as a decode request with key splits does.
//
// Persistent: one CTA per SM walks the units the host dealt it; the K/V rings
// are indexed by a tile counter that runs across units.
//
// Warp roles (384 threads; the register split and warps 12-15 or 12-19 over
// E4M3 pools are described next to the kernel's configuration):
//   warp 8      TMA producer: each unit's Q of both blocks (3-D boxes
//               [bq][G][64], one per quadrant and column half) after the unit's
//               first K/V tile, and the prompt K/V tiles into a KST-deep K ring
//               and a VST-deep V ring (one 2-D box of min(page, 64) rows x 64
//               columns per page slice, column half and tensor). It is the one
//               waiter on the slot-release barriers, taking every tile's release
//               in order (a parity wait only names the right phase for a waiter
//               that is never two phases behind); a tail tile's slots it hands
//               to warps 10-11 by raising a shared counter;
//   warp 9      TMEM allocation; one thread issues tcgen05.mma in the order
//               Q K_t^T -> S_A, Q K_t^T -> S_B, P_A V_t -> O_A, Q K_{t+1}^T -> S_A,
//               P_B V_t -> O_B, Q K_{t+1}^T -> S_B, ...: while the softmax warps of
//               one block work on their scores, the tensor core serves the other;
//   warps 0-3   softmax of block A, warps 4-7 softmax of block B: thread <->
//               query row <-> TMEM lane; scores read from TMEM twice (row
//               maximum, then probabilities), online softmax in base 2 with a
//               lazy rescale of O (only when a row maximum grows by more than
//               2^8), P written as 16-bit pairs over the first 64 columns of the
//               block's S; at the end of a unit the same warps normalise O and
//               write it (final O and LSE, or the fp32 partial state);
//   warps 10-11 tail tiles: resolve a unit's tail keys one unit ahead (and
//               bring their rows into L2), then copy K and V rows into the ring
//               slots with 16-byte cp.async in the 128-byte-swizzled layout a
//               TMA box would have (absent keys are zero rows), with a key ->
//               pool-row table per V slot for the softmax's mask;
//   warps 12-19 (E4M3 pools only, 640 threads): the producer loads each E4M3
//               tile into the upper half of its 16-bit ring slot; warps 12-15
//               widen every K tile, warps 16-19 every V tile, in place, to the
//               q dtype, and complete the slot's full barrier (two streams, so
//               a late V tile does not hold the next K tile back).
// TMEM columns: S_A [0, 128), S_B [128, 256), O_A [256, 256 + D), O_B after it.
// One S per block: Q K_{t+1}^T into S_X is issued after P_X V_t, and
// tcgen05.mma instructions of one thread execute in issue order, so P_t (which
// aliases S_X) is read before it is overwritten; the completion of Q K_{t+1}^T
// also implies that of P_X V_t, which is what a rescale of O_X needs.
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
namespace {

template <int D>
struct WideCfg {
    static constexpr int TK = 128;                          // keys per tile
    static constexpr int NC = D / 64;                       // 128-byte column regions per row
    static constexpr int Q_BYTES = kRowsPerBlock * D * 2;   // one block's Q: NC regions of 128 rows x 128 B
    static constexpr int KV_BYTES = TK * D * 2;             // one K (or V) tile
    static constexpr int KST = D == 64 ? 5 : 2;             // K ring depth
    static constexpr int VST = D == 64 ? 6 : 3;             // V ring depth
    static constexpr int OFF_K = 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
    static constexpr int OFF_TROW = OFF_V + VST * KV_BYTES;  // int [VST][TK]: pool row of tail key c, -1: none
    static constexpr int OFF_BAR = OFF_TROW + VST * TK * 4;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;        // barriers + alignment slack
    static constexpr int S_COL = 0;                          // S of block X: [X * TK, X * TK + TK)
    static constexpr int O_COL = 2 * TK;                     // O of block X: [O_COL + X * D, + D)
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 384;
    static constexpr int GATHER_TID0 = 320;                  // warps 10-11
    // over E4M3 pools eight more warps (12-19, two warpgroups) widen the prompt tiles: warps 12-15 every K
    // tile, warps 16-19 every V tile, two streams that do not wait on each other. Registers per thread:
    // 96 at launch (__launch_bounds__(640, 1)), then the widening warps down to REGS_CONV and the softmax
    // warps (0-7) up to REGS_SOFTMAX (setmaxnreg draws on the launch's registers; warps 8-11 keep 96)
    static constexpr int THREADS_E4M3 = 640;
    static constexpr int CONV_TID0 = 384;
    static constexpr int CONV_THREADS = 128;  // per stream
    static constexpr int REGS_LAUNCH_E4M3 = 96;
    static constexpr int REGS_CONV = 64;
    static constexpr int REGS_SOFTMAX = 128;
    static_assert(256 * REGS_SOFTMAX + 128 * REGS_LAUNCH_E4M3 + 256 * REGS_CONV <= THREADS_E4M3 * REGS_LAUNCH_E4M3,
                  "register split");
    static_assert(O_COL + 2 * D <= 512, "tensor memory");
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(KST <= 8 && VST <= 8, "barrier arrays");
    static_assert(KST >= 2 && VST >= 2, "ring depth (one slot would stall the next tile's loads)");
};

struct WideBarriers {
    uint64_t k_full[8];
    uint64_t k_empty[8];   // both blocks' Q*K^T of the tile completed (arrived by block B's warp 6)
    uint64_t v_full[8];
    uint64_t v_empty[8];   // both blocks' P*V of the tile completed (arrived by block B's warp 6 with the next
                           // tile's S_B)
    uint64_t q_full[2];    // block X's Q of a unit landed
    uint64_t q_empty[2];   // ... and the unit's last Q*K^T of block X completed
    uint64_t s_full[2];    // Q*K^T into S_X completed
    uint64_t p_full[2];    // block X's softmax warps wrote P_X (one arrival per warp)
    uint64_t o_final[2];   // the last P*V of a unit into O_X completed
    uint64_t drain;
    uint64_t k8_full[8];   // E4M3 pools: the E4M3 K tile landed in the upper half of the K slot
    uint64_t v8_full[8];   // ... the E4M3 V tile in the V slot
    uint32_t tmem_base;
    int abort_flag;
    int tail_granted;      // tail tiles whose ring slots the producer has handed to the tail-tile warps
};

constexpr uint64_t kWideWaitNs = 1000000000ull;  // 1 s without progress
constexpr uint64_t kWideDrainNs = 200000000ull;

// tail tiles of a unit: the request's W * T tail keys, beam-major, in tiles of 128 keys
__device__ __forceinline__ int wide_tail_tiles(const UnitInfo& ui) {
    return (ui.fused && ui.T > 0) ? (ui.rows * ui.T + 127) / 128 : 0;
}

// Named barrier `id` over `n` threads, returning the AND of their flags. Every one of them takes part in
// every call (a flag that is false makes them all stop together).
__device__ __forceinline__ bool named_sync_and(int id, int n, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(ok)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
// Named barrier 1 over the 64 tail-tile threads, returning the AND of their flags. Every one of them
// takes part in every call (a flag that is false makes them all stop together).
__device__ __forceinline__ bool gather_sync_and(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 64, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(ok))
        : "memory");
    return r != 0;
}

}  // namespace

template <int D, bool BF16, bool FP8>
__global__ void __launch_bounds__(FP8 ? 640 : 384, 1)
prefix_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefixParams p) {
    using C = WideCfg<D>;
    constexpr int TK = C::TK, NC = C::NC, KST = C::KST, VST = C::VST;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto q_buf = [&](int x) -> uint8_t* { return smem + x * C::Q_BYTES; };
    auto k_tile = [&](int gt) -> uint8_t* { return smem + C::OFF_K + (gt % KST) * C::KV_BYTES; };
    auto v_tile = [&](int gt) -> uint8_t* { return smem + C::OFF_V + (gt % VST) * C::KV_BYTES; };
    auto trow_of = [&](int gt) -> int* { return reinterpret_cast<int*>(smem + C::OFF_TROW) + (gt % VST) * TK; };
    WideBarriers* bars = reinterpret_cast<WideBarriers*>(smem + C::OFF_BAR);
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
    const int qrows = p.bq * p.G;  // rows a quadrant's TMA box fills

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
            mbar_init(&bars->q_empty[i], 1);
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->p_full[i], 4);  // one arrival per softmax warp of the block
            mbar_init(&bars->o_final[i], 1);
        }
        mbar_init(&bars->drain, 1);
        if constexpr (FP8) {
            for (int s = 0; s < KST; ++s) mbar_init(&bars->k8_full[s], 1);
            for (int s = 0; s < VST; ++s) mbar_init(&bars->v8_full[s], 1);
        }
        bars->abort_flag = 0;
        bars->tail_granted = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 9) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
    // zero the query rows no TMA box covers (rows bq * G .. 31 of each quadrant of both blocks), so
    // padded rows stay finite
    {
        constexpr int NCHUNK = 2 * NC * kRowsPerBlock * 8;  // 16-byte chunks of the two Q buffers
        for (int idx = tid; idx < NCHUNK; idx += (FP8 ? C::THREADS_E4M3 : C::THREADS)) {
            const int r = (idx >> 3) & (kRowsPerBlock - 1);
            if ((r & 31) >= qrows) reinterpret_cast<uint4*>(smem)[idx] = make_uint4(0, 0, 0, 0);
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

    if (warp >= 8) {
        // over E4M3 pools the widening warps (12-19, two warpgroups) give registers to the softmax
        // warpgroups
        if constexpr (FP8) {
            if (warp >= 12) setmaxnreg_dec<C::REGS_CONV>();
        }
        if (warp == 8) {
            // ================= TMA producer =================
            const int BR = ps < kTileKeys ? ps : kTileKeys;  // rows per box (a page, or 64 rows of a larger page)
            int gt = 0, k = 0, ntail = 0;
            bool ok = true;
            for (int u = u_begin; u < u_end && ok; ++u, ++k) {
                const UnitInfo ui = load_unit(p, u);
                const int ptiles = prompt_tiles<TK>(ui);
                const int ntiles = ptiles + wide_tail_tiles(ui);
                const int* pg = p.pages + ui.page_off;
                const int npages = (ui.P + ps - 1) >> p.ps_log2;
                int win_base = -1, my_page = 0;
                for (int t = 0; t < ntiles; ++t, ++gt) {
                    // this warp is the only waiter on the slot-release barriers and takes every tile's
                    // release in order, so each parity wait names the phase it means
                    if (gt >= KST) {
                        ok = mbar_wait(&bars->k_empty[gt % KST], ((gt / KST) - 1) & 1, abort_flag, kWideWaitNs);
                        ok = __all_sync(FULL, ok);
                        if (!ok) break;
                    }
                    if (t >= ptiles) {
                        // a tail tile: once its V slot is free too, hand both slots to the tail-tile warps
                        // (a counter, not a barrier phase: they may lag several tail tiles behind)
                        if (gt >= VST) {
                            ok = mbar_wait(&bars->v_empty[gt % VST], ((gt / VST) - 1) & 1, abort_flag, kWideWaitNs);
                            ok = __all_sync(FULL, ok);
                            if (!ok) break;
                        }
                        ++ntail;
                        if (lane == 0) {
                            counter_release(&bars->tail_granted, ntail);
                            if constexpr (FP8) {
                                // no E4M3 tile here: complete the slots' E4M3 phases (the widening warps wait
                                // for every phase in order and have nothing to widen for a tail tile), so that
                                // the phases keep counting the slot's tiles
                                mbar_arrive(&bars->k8_full[gt % KST]);
                                mbar_arrive(&bars->v8_full[gt % VST]);
                            }
                        }
                        __syncwarp();
                        continue;
                    }
                    const int key0 = ui.key_begin + t * TK;
                    const int valid = min(TK, ui.key_end - key0);
                    const int nchunks = (valid + BR - 1) / BR;  // pages (or 64-row slices) with valid keys
                    const int tile_bytes = nchunks * BR * D * (FP8 ? 1 : 2);
                    const int pidx0 = key0 >> p.ps_log2;
                    const int pidx_last = (key0 + (nchunks - 1) * BR) >> p.ps_log2;
                    if (win_base < 0 || pidx_last >= win_base + 32) {  // warp-uniform
                        win_base = pidx0;
                        my_page = (win_base + lane < npages) ? __ldg(pg + win_base + lane) : 0;
                    }
                    // box b of a tensor: column half b % NC of chunk b / NC (E4M3: one box of head_dim bytes
                    // per chunk, into the upper half of the slot, where the widening warps pick it up)
                    constexpr int NB = FP8 ? 1 : NC;
                    const int nbox = nchunks * NB;
                    for (int tensor = 0; tensor < 2; ++tensor) {
                        if (tensor == 1 && gt >= VST) {
                            ok = mbar_wait(&bars->v_empty[gt % VST], ((gt / VST) - 1) & 1, abort_flag, kWideWaitNs);
                            ok = __all_sync(FULL, ok);
                            if (!ok) break;
                        }
                        uint64_t* full = FP8 ? (tensor == 0 ? &bars->k8_full[gt % KST] : &bars->v8_full[gt % VST])
                                             : (tensor == 0 ? &bars->k_full[gt % KST] : &bars->v_full[gt % VST]);
                        uint8_t* base = tensor == 0 ? k_tile(gt) : v_tile(gt);
                        const CUtensorMap* map = tensor == 0 ? &tm_k : &tm_v;
                        if (lane == 0) mbar_arrive_expect_tx(full, tile_bytes);
                        for (int b0 = 0; b0 < nbox; b0 += 32) {
                            const int bx = b0 + lane;
                            const int ch = min(bx / NB, nchunks - 1);
                            const int key = key0 + ch * BR;
                            int page = __shfl_sync(FULL, my_page, (key >> p.ps_log2) - win_base);
                            if (bx < nbox) {
                                if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
                                    atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
                                    page = 0;
                                }
                                const int row = ((page * p.Hkv + ui.g) << p.ps_log2) + (key & (ps - 1));
                                if constexpr (FP8) {
                                    tma_load_2d(base + TK * D + ch * BR * D, map, full, 0, row);
                                } else {
                                    const int c = bx % NC;
                                    tma_load_2d(base + c * TK * 128 + ch * BR * 128, map, full, c * 64, row);
                                }
                            }
                        }
                    }
                    if (!ok) break;
                    if (t == 0) {
                        // the unit's Q of both blocks, once the previous unit's last Q*K^T of the block is done
                        // (issued after this unit's first K/V tile, which may already stream meanwhile)
                        for (int x = 0; x < 2 && ok; ++x) {
                            if (k >= 1) {
                                ok = mbar_wait(&bars->q_empty[x], (k - 1) & 1, abort_flag, kWideWaitNs);
                                ok = __all_sync(FULL, ok);
                                if (!ok) break;
                            }
                            if (lane == 0) {
                                mbar_arrive_expect_tx(&bars->q_full[x], NC * 4 * qrows * 128);
                                for (int c = 0; c < NC; ++c)
                                    for (int i = 0; i < 4; ++i)
                                        tma_load_3d(q_buf(x) + c * (kRowsPerBlock * 128) + i * 32 * 128, &tm_q,
                                                    &bars->q_full[x], c * 64, ui.g * p.G,
                                                    ui.row_off + (2 * ui.rb + x) * p.Wblk + i * p.bq);
                            }
                        }
                        if (!ok) break;
                    }
                    __syncwarp();
                }
            }
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
                }
                // drain: let this CTA's own copies land before the CTA exits
                // (the TMA loads complete the E4M3 barriers over E4M3 pools)
                const uint64_t t0 = globaltimer_ns();
                uint64_t* kf = FP8 ? bars->k8_full : bars->k_full;
                uint64_t* vf = FP8 ? bars->v8_full : bars->v_full;
                for (int j = max(0, gt - KST); j <= gt; ++j)
                    while (!mbar_try_wait(&kf[j % KST], (j / KST) & 1) && globaltimer_ns() - t0 < kWideDrainNs) {
                    }
                for (int j = max(0, gt - VST); j <= gt; ++j)
                    while (!mbar_try_wait(&vf[j % VST], (j / VST) & 1) && globaltimer_ns() - t0 < kWideDrainNs) {
                    }
                for (int x = 0; x < 2; ++x)
                    while (!mbar_try_wait(&bars->q_full[x], k & 1) && globaltimer_ns() - t0 < kWideDrainNs) {
                    }
            }
        } else if (warp == 9) {
            // ================= MMA issuer =================
            if (lane == 0) {
                constexpr uint32_t ID_QK = idesc_f16(kRowsPerBlock, TK, BF16, false);
                constexpr uint32_t ID_PV = idesc_f16(kRowsPerBlock, D, BF16, true);
                int gt = 0, k = 0;
                int pend = -1;  // tile whose P*V is not issued yet
                bool pend_first = false, pend_last = false;
                bool ok = true;
                // (V of tile j is waited for before block A's P: a wait that has already completed still costs
                // a shared-memory round trip, which would otherwise sit between P and the MMAs)
                auto issue_pv = [&](int x, int j, bool first, bool last) -> bool {
                    if (!mbar_wait(&bars->p_full[x], j & 1, abort_flag, kWideWaitNs)) return false;
                    tc_fence_after();
                    const uint32_t p_tmem = tmem + C::S_COL + x * TK;
                    const uint32_t o_tmem = tmem + C::O_COL + x * D;
                    const uint32_t v_addr = smem_u32(v_tile(j));
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk) {
                        const uint64_t bd = sdesc_sw128(v_addr + kk * 16 * 128, TK * 128, 1024);
                        mma_f16_tmem_a(o_tmem, p_tmem + kk * 8, bd, ID_PV, (!first || kk > 0) ? 1u : 0u);
                    }
                    if (last) mma_commit(&bars->o_final[x]);
                    return true;
                };
                for (int u = u_begin; u < u_end && ok; ++u, ++k) {
                    const UnitInfo ui = load_unit(p, u);
                    const int ntiles = prompt_tiles<TK>(ui) + wide_tail_tiles(ui);
                    for (int t = 0; t < ntiles; ++t, ++gt) {
                        const uint32_t k_addr = smem_u32(k_tile(gt));
                        // the loads this tile's MMAs need, first: they do not depend on the softmax, and once
                        // a block's P is ready its P*V and the next Q*K^T go out back to back
                        ok = mbar_wait(&bars->k_full[gt % KST], (gt / KST) & 1, abort_flag, kWideWaitNs);
                        if (ok && t == 0) ok = mbar_wait(&bars->q_full[0], k & 1, abort_flag, kWideWaitNs);
                        if (ok && t == 0) ok = mbar_wait(&bars->q_full[1], k & 1, abort_flag, kWideWaitNs);
                        if (ok && pend >= 0)
                            ok = mbar_wait(&bars->v_full[pend % VST], (pend / VST) & 1, abort_flag, kWideWaitNs);
                        if (!ok) break;
                        for (int x = 0; x < 2; ++x) {
                            if (pend >= 0) {
                                ok = issue_pv(x, pend, pend_first, pend_last);
                                if (!ok) break;
                            }
                            // S_X holds P_X of the previous tile, whose P*V was issued just before
                            tc_fence_after();
                            const uint32_t q_addr = smem_u32(q_buf(x));
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint64_t ad =
                                    sdesc_sw128(q_addr + (kk >> 2) * (kRowsPerBlock * 128) + (kk & 3) * 32, 16, 1024);
                                const uint64_t bd = sdesc_sw128(k_addr + (kk >> 2) * (TK * 128) + (kk & 3) * 32, 16, 1024);
                                mma_f16(tmem + C::S_COL + x * TK, ad, bd, ID_QK, kk > 0 ? 1u : 0u);
                            }
                            // (the K and V slots are released by block B's softmax warp 6 once it sees S_B
                            // complete)
                            mma_commit(&bars->s_full[x]);
                            if (t == ntiles - 1) mma_commit(&bars->q_empty[x]);
                        }
                        if (!ok) break;
                        pend = gt;
                        pend_first = t == 0;
                        pend_last = t == ntiles - 1;
                    }
                }
                if (ok && pend >= 0) {
                    ok = mbar_wait(&bars->v_full[pend % VST], (pend / VST) & 1, abort_flag, kWideWaitNs);
                    if (ok) ok = issue_pv(0, pend, pend_first, pend_last);
                    if (ok) ok = issue_pv(1, pend, pend_first, pend_last);
                }
                if (!ok) {
                    *abort_flag = 1;
                    atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
                }
                // drain: every MMA issued by this thread completes before TMEM is freed
                mma_commit(&bars->drain);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&bars->drain, 0) && globaltimer_ns() - t0 < kWideDrainNs) {
                }
            }
        } else if (warp < 12) {
            // ================= tail tiles =================
            constexpr int CH = D / 8;     // 16-byte chunks of a 16-bit K or V row
            constexpr int RPS = 64 / CH;  // rows one pass of the 64 threads covers
            constexpr int EB = FP8 ? 1 : 2;  // bytes per pool element
            const int gtid = tid - C::GATHER_TID0;
            const int kc = gtid % CH;
            const int rsub = gtid / CH;
            const uint8_t* k_pool = static_cast<const uint8_t*>(p.k_pool);
            const uint8_t* v_pool = static_cast<const uint8_t*>(p.v_pool);
            // pool rows of this thread's two key columns (gtid, gtid + 64) of each tail tile of a unit,
            // resolved a unit ahead; -1 past the request's tail keys or when unreadable
            int res[kWideMaxTailTiles][2];
            auto resolve = [&](const UnitInfo& ui) {
                const int ntt = wide_tail_tiles(ui);
#pragma unroll
                for (int n = 0; n < kWideMaxTailTiles; ++n)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        res[n][h] = -1;
                        const int cc = n * TK + gtid + 64 * h;
                        if (n >= ntt || cc >= ui.rows * ui.T) continue;
                        const int w = cc / ui.T, tt = cc - w * ui.T;
                        const int pos = ui.P + tt;
                        const int src = __ldg(p.ci + (static_cast<long long>(ui.b) * p.W + w) * p.max_seq + pos);
                        int r = -1;
                        if (static_cast<unsigned>(src) < static_cast<unsigned>(p.W)) {
                            const int page = __ldg(p.beam_pages +
                                                   (static_cast<long long>(ui.b) * p.W + src) * p.beam_pages_stride +
                                                   (pos >> p.ps_log2));
                            if (static_cast<unsigned>(page) < static_cast<unsigned>(p.num_pages))
                                r = ((page * p.Hkv + ui.g) << p.ps_log2) + (pos & (ps - 1));
                        }
                        if (r < 0) {
                            atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
                        } else {
                            // the gather runs at the end of the unit: bring the row's K and V into L2 now
#pragma unroll
                            for (int off = 0; off < D * EB; off += 128) {
                                prefetch_l2(k_pool + static_cast<long long>(r) * (D * EB) + off);
                                prefetch_l2(v_pool + static_cast<long long>(r) * (D * EB) + off);
                            }
                        }
                        res[n][h] = r;
                    }
            };
            bool ok = true;
            int gt = 0, ntail = 0;
            UnitInfo cur;
            if (nunits > 0) {
                cur = load_unit(p, u_begin);
                resolve(cur);
            }
            for (int k = 0; k < nunits && ok; ++k) {
                const int ptiles = prompt_tiles<TK>(cur);
                const int ntt = wide_tail_tiles(cur);
#pragma unroll
                for (int n = 0; n < kWideMaxTailTiles; ++n) {
                    if (n >= ntt) break;
                    const int gtt = gt + ptiles + n;
                    // the producer hands the tile's K and V slots over once both blocks' Q*K^T and P*V of
                    // their previous tiles are done
                    ok = counter_wait(&bars->tail_granted, ntail, abort_flag, kWideWaitNs);
                    ++ntail;
                    ok = __all_sync(FULL, ok);
                    int* trow = trow_of(gtt);
                    if (ok) {
                        trow[gtid] = res[n][0];
                        trow[gtid + 64] = res[n][1];
                    }
                    ok = gather_sync_and(ok);
                    if (ok) {
                        uint8_t* kt = k_tile(gtt);
                        uint8_t* vt = v_tile(gtt);
#pragma unroll 4
                        for (int i = 0; i < TK / RPS; ++i) {
                            const int c = rsub + i * RPS;
                            const int r = trow[c];
                            // the layout of a TMA box with 128-byte swizzle: chunk kc of row c in column half kc / 8
                            const uint32_t off = sw128_chunk<TK>(kc, c);
                            const long long e = static_cast<long long>(r < 0 ? 0 : r) * D + kc * 8;  // element offset
                            if constexpr (FP8) {
                                uint4 kw = make_uint4(0, 0, 0, 0), vw = kw;  // absent keys are zero rows
                                if (r >= 0) {
                                    kw = e4m3x8_to_16<BF16>(__ldg(reinterpret_cast<const uint2*>(k_pool + e)));
                                    vw = e4m3x8_to_16<BF16>(__ldg(reinterpret_cast<const uint2*>(v_pool + e)));
                                }
                                *reinterpret_cast<uint4*>(kt + off) = kw;
                                *reinterpret_cast<uint4*>(vt + off) = vw;
                            } else {
                                const uint32_t nb = r < 0 ? 0u : 16u;  // absent keys are zero rows
                                cp_async16(kt + off, k_pool + 2 * e, nb);
                                cp_async16(vt + off, v_pool + 2 * e, nb);
                            }
                        }
                        if constexpr (!FP8) cp_async_commit_wait_all();
                        fence_proxy_async_smem();
                    }
                    ok = gather_sync_and(ok);
                    if (!ok) break;
                    if (gtid == 0) {
                        mbar_arrive(&bars->k_full[gtt % KST]);
                        mbar_arrive(&bars->v_full[gtt % VST]);
                    }
                }
                gt += ptiles + ntt;
                if (ok && k + 1 < nunits) {
                    cur = load_unit(p, u_begin + k + 1);
                    resolve(cur);
                }
            }
            if (!ok && gtid == 0) {
                *abort_flag = 1;
                atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
            }
        } else {
            // ================= E4M3 pools: widening of the prompt tiles (warps 12-15) =================
            if constexpr (FP8) {
                const int ctid = tid - C::CONV_TID0;
                const int tensor = ctid / C::CONV_THREADS;  // 0: K tiles (warps 12-15), 1: V tiles (warps 16-19)
                const int stid = ctid % C::CONV_THREADS;
                const int bar = 2 + tensor;                 // named barrier of the stream's threads
                bool ok = true;
                int gt = 0;
                for (int k = 0; k < nunits && ok; ++k) {
                    const UnitInfo cur = load_unit(p, u_begin + k);
                    const int ptiles = prompt_tiles<TK>(cur);
                    const int ntiles = ptiles + wide_tail_tiles(cur);
                    for (int t = 0; t < ntiles && ok; ++t, ++gt) {
                        // every tile's E4M3 phase in order, a tail tile's too (the producer completes it when it
                        // hands the slots over; nothing to widen): so each parity wait names the phase it means
                        uint64_t* full8 = tensor == 0 ? &bars->k8_full[gt % KST] : &bars->v8_full[gt % VST];
                        const uint32_t ph = tensor == 0 ? (gt / KST) & 1 : (gt / VST) & 1;
                        ok = mbar_wait(full8, ph, abort_flag, kWideWaitNs);
                        ok = __all_sync(FULL, ok);
                        ok = named_sync_and(bar, C::CONV_THREADS, ok);
                        if (!ok || t >= ptiles) continue;
                        const int valid = min(TK, cur.key_end - (cur.key_begin + t * TK));
                        widen_e4m3_tile<D, TK, BF16, C::CONV_THREADS>(tensor == 0 ? k_tile(gt) : v_tile(gt), valid,
                                                                      stid, bar);
                        fence_proxy_async_smem();
                        ok = named_sync_and(bar, C::CONV_THREADS, ok);
                        if (ok && stid == 0)
                            mbar_arrive(tensor == 0 ? &bars->k_full[gt % KST] : &bars->v_full[gt % VST]);
                    }
                }
                if (!ok && stid == 0) {
                    *abort_flag = 1;
                    atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
                }
            }
        }
    } else {
        if constexpr (FP8) setmaxnreg_inc<C::REGS_SOFTMAX>();
        // ================= softmax warps (block x), then the unit's output =================
        const int x = warp >> 2;
        const int quad = warp & 3;           // TMEM lane quadrant this warp may access
        const int wq = lane / p.G;           // beam of the quadrant
        const int jh = lane - wq * p.G;      // head of the group
        const int wbl = quad * p.bq + wq;    // beam of the block
        const bool row_ok = lane < qrows;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t s_col = lane_base + C::S_COL + x * TK;
        const uint32_t o_col = lane_base + C::O_COL + x * D;
        const float sl2 = p.scale_log2;
        const uint32_t ninf = __float_as_uint(-INFINITY);
        bool ok = true;
        int gt = 0;
        for (int k = 0; k < nunits && ok; ++k) {
            const UnitInfo cur = load_unit(p, u_begin + k);
            const int ptiles = prompt_tiles<TK>(cur);
            const int ntiles = ptiles + wide_tail_tiles(cur);
            // the block's first beam (prompt token of a prefill: units of two blocks each)
            const int w0 = (2 * cur.rb + x) * p.Wblk;
            const int wb = w0 + wbl;                    // beam of the request
            const int nw = min(p.Wblk, cur.rows - w0);  // beams of this block (<= 0: none)
            const bool live = row_ok && wbl < nw;
            // a warp whose rows are all padding skips the arithmetic but keeps the barrier protocol
            const bool warp_live = quad * p.bq < nw;
            float m = -INFINITY, l = 0.f;
            for (int t = 0; t < ntiles; ++t, ++gt) {
                const bool tail = t >= ptiles;
                const int valid = tail ? TK : min(TK, cur.key_end - (cur.key_begin + t * TK));
                ok = mbar_wait(&bars->s_full[x], gt & 1, abort_flag, kWideWaitNs);
                // S_B complete: every MMA the issuing thread issued before Q*K_gt^T -> S_B has completed:
                // both blocks' Q*K^T of this tile and both blocks' P*V of the previous one. One thread of
                // block B hands the K slot of this tile and the V slot of the previous tile back to the
                // producer (no further commits in the MMA thread: a commit right after another holds the
                // issuing thread until the first one's MMAs finish)
                if (ok && warp == 6 && lane == 0) {
                    mbar_arrive(&bars->k_empty[gt % KST]);
                    if (gt >= 1) mbar_arrive(&bars->v_empty[(gt - 1) % VST]);
                }
                // a tail tile's key table is complete once its V slot is full
                if (ok && tail) ok = mbar_wait(&bars->v_full[gt % VST], (gt / VST) & 1, abort_flag, kWideWaitNs);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc_fence_after();
                if (warp_live) {
                    // masked keys count as -inf: no part in the maximum, probability exp2(-inf) = 0. A
                    // partial prompt tile keeps [0, valid); a tail tile keeps the row's own beam's T
                    // columns (w * T - first column of the tile, T <= 8: at most two 32-bit words) whose
                    // key is readable
                    // a causal prefill row t sees keys 0 .. C + t: its own count of valid keys in this tile
                    int rvalid = valid;
                    if (cur.causal >= 0) rvalid = min(valid, cur.causal + wb + 1 - (cur.key_begin + t * TK));
                    const bool partial = valid < TK || tail || (cur.causal >= 0 && __any_sync(FULL, rvalid < TK));
                    uint32_t km[TK / 32];
                    if (partial) {
                        if (tail) {
                            uint64_t win = 0;
                            int wbase = 0;
                            if (live) {
                                const int lo = wb * cur.T - (t - ptiles) * TK;
                                const int c0 = max(lo, 0), c1 = min(lo + cur.T, TK);
                                wbase = c0 & ~31;
                                const int* trow = trow_of(gt);
                                for (int c = c0; c < c1; ++c)
                                    if (trow[c] >= 0) win |= 1ull << (c - wbase);
                            }
#pragma unroll
                            for (int j = 0; j < TK / 32; ++j)
                                km[j] = 32 * j == wbase        ? static_cast<uint32_t>(win)
                                        : 32 * j == wbase + 32 ? static_cast<uint32_t>(win >> 32)
                                                               : 0u;
                        } else {
#pragma unroll
                            for (int j = 0; j < TK / 32; ++j) {
                                const int n = min(max(rvalid - 32 * j, 0), 32);
                                km[j] = n == 32 ? ~0u : (1u << n) - 1u;
                            }
                        }
                    }
                    auto mask_pair = [&](int c0, uint32_t& ma, uint32_t& mb) {
                        ma = c0 == 0 ? km[0] : km[2];
                        mb = c0 == 0 ? km[1] : km[3];
                    };
                    // pass 1: the row maximum of the raw scores, then scaled (the scale is positive)
                    float mp[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) mp[j] = -INFINITY;
                    float mred = -INFINITY;
#pragma unroll 1
                    for (int c0 = 0; c0 < TK; c0 += 64) {
                        uint32_t ma = ~0u, mb = ~0u;
                        if (partial) {
                            mask_pair(c0, ma, mb);
                            if (!__any_sync(FULL, (ma | mb) != 0u)) continue;  // no row of the warp keeps one
                        }
                        uint32_t sa[32], sb[32];
                        if (!partial) {
                            // the loads reduce each 32-column half to its maximum
                            float ra, rb;
                            tmem_ld32_max(s_col + c0, sa, ra);
                            tmem_ld32_max(s_col + c0 + 32, sb, rb);
                            tmem_wait_ld();
                            mred = fmax3(mred, ra, rb);
                            continue;
                        }
                        tmem_ld32(s_col + c0, sa);
                        tmem_ld32(s_col + c0 + 32, sb);
                        tmem_wait_ld();
                        if (__any_sync(FULL, (ma & mb) != ~0u)) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                sa[c] = (ma >> c) & 1u ? sa[c] : ninf;
                                sb[c] = (mb >> c) & 1u ? sb[c] : ninf;
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            mp[c & 7] = fmax3(mp[c & 7], __uint_as_float(sa[c]), __uint_as_float(sb[c]));
                    }
                    const float mxr = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]),
                                            fmax3(mp[6], mp[7], mred));
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
                        // P_X V of the previous tile has completed (it was issued before the Q*K^T whose
                        // completion s_full reported), and this tile's P*V waits for p_full
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t orr[32];
                            tmem_ld32(o_col + c0, orr);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                            tmem_st32(o_col + c0, orr);
                        }
                    }
                    // pass 2: probabilities 2^(s * scale_log2 - m) and their sum; P in 16-bit pairs over
                    // the first 64 columns of S_X, 64 keys per store (P columns [32i, 32i + 32) overwrite
                    // score columns already read in this pass)
                    const float nm = -m;
                    float rsp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                    for (int c0 = 0; c0 < TK; c0 += 64) {
                        uint32_t ma = ~0u, mb = ~0u;
                        if (partial) mask_pair(c0, ma, mb);
                        uint32_t pk[32];
                        if (partial && !__any_sync(FULL, (ma | mb) != 0u)) {
#pragma unroll
                            for (int c = 0; c < 32; ++c) pk[c] = 0u;
                            tmem_st32(s_col + (c0 >> 1), pk);
                            continue;
                        }
                        uint32_t sa[32], sb[32];
                        tmem_ld32(s_col + c0, sa);
                        tmem_ld32(s_col + c0 + 32, sb);
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
                            float e0, e1, e2, e3;
                            fma2_bc(e0, e1, __uint_as_float(sa[c]), __uint_as_float(sa[c + 1]), sl2, nm);
                            fma2_bc(e2, e3, __uint_as_float(sb[c]), __uint_as_float(sb[c + 1]), sl2, nm);
                            const float p0 = exp2f(e0), p1 = exp2f(e1), p2 = exp2f(e2), p3 = exp2f(e3);
                            add2_acc(rsp[0], rsp[1], p0, p1);
                            add2_acc(rsp[2], rsp[3], p2, p3);
                            pk[c >> 1] = pack2<BF16>(p0, p1);
                            pk[16 + (c >> 1)] = pack2<BF16>(p2, p3);
                        }
                        tmem_st32(s_col + (c0 >> 1), pk);
                    }
                    tmem_wait_st();
                    l += (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
                }
                if (!FP8 && x == 0 && !tail && valid < TK) {
                    // a unit's last prompt tile: zero V rows past the valid keys (stale or garbage rows
                    // times P = 0 must not produce NaN); block A's warps, before block A's P*V, which the
                    // tensor core issues before block B's
                    ok = mbar_wait(&bars->v_full[gt % VST], (gt / VST) & 1, abort_flag, kWideWaitNs);
                    ok = __all_sync(FULL, ok);
                    if (!ok) break;
                    uint8_t* sV = v_tile(gt);
                    const int nzc = (TK - valid) * 8;  // 16-byte chunks per column half
                    for (int c = 0; c < NC; ++c)
                        for (int idx = tid; idx < nzc; idx += 128)
                            reinterpret_cast<uint4*>(sV + c * TK * 128 + valid * 128)[idx] = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[x]);
            }
            if (!ok) break;
            // ---- the unit's output: O_X once its last P*V has completed. The next unit's first P*V
            // (which overwrites O_X) waits for this warp's next p_full arrival, after these reads.
            ok = mbar_wait(&bars->o_final[x], k & 1, abort_flag, kWideWaitNs);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc_fence_after();
            if (warp_live) {
                const float inv = p.v_scale / l;  // the values' E4M3 scale (1 over 16-bit pools)
                if (cur.fused) {
                    // the request's whole key set went through this unit: the final O (q dtype) and LSE
                    const long long rh = (static_cast<long long>(cur.row_off) + wb) * p.Hq + cur.g * p.G + jh;
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + rh * D);
                    // rows start at multiples of 128 bytes: 32-byte stores when o is 32-byte aligned
                    const bool st32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t orr[32];
                        tmem_ld32(o_col + c0, orr);
                        tmem_wait_ld();
                        if (live) {
                            uint4 w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float* f = reinterpret_cast<const float*>(orr) + 8 * e;
                                w[e] = make_uint4(pack2<BF16>(f[0] * inv, f[1] * inv), pack2<BF16>(f[2] * inv, f[3] * inv),
                                                  pack2<BF16>(f[4] * inv, f[5] * inv), pack2<BF16>(f[6] * inv, f[7] * inv));
                            }
                            if (st32) {
                                st_global_v8(dst + (c0 >> 3), w[0], w[1]);
                                st_global_v8(dst + (c0 >> 3) + 2, w[2], w[3]);
                            } else {
#pragma unroll
                                for (int e = 0; e < 4; ++e) dst[(c0 >> 3) + e] = w[e];
                            }
                        }
                    }
                    if (live) {
                        const float lse2 = m + log2f(l);
                        p.lse[rh] = p.lse_base2 ? lse2 : lse2 * 0.69314718055994530942f;
                    }
                } else {
                    const long long prow = (static_cast<long long>(cur.part) * p.W + wb) * p.Hq + cur.g * p.G + jh;
                    float4* dst = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t orr[32];
                        tmem_ld32(o_col + c0, orr);
                        tmem_wait_ld();
                        if (live) {
                            // (the workspace's partial rows are 32-byte aligned)
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const uint4 lo = make_uint4(__float_as_uint(__uint_as_float(orr[4 * e]) * inv),
                                                            __float_as_uint(__uint_as_float(orr[4 * e + 1]) * inv),
                                                            __float_as_uint(__uint_as_float(orr[4 * e + 2]) * inv),
                                                            __float_as_uint(__uint_as_float(orr[4 * e + 3]) * inv));
                                const uint4 hi = make_uint4(__float_as_uint(__uint_as_float(orr[4 * e + 4]) * inv),
                                                            __float_as_uint(__uint_as_float(orr[4 * e + 5]) * inv),
                                                            __float_as_uint(__uint_as_float(orr[4 * e + 6]) * inv),
                                                            __float_as_uint(__uint_as_float(orr[4 * e + 7]) * inv));
                                st_global_v8(dst + (c0 >> 2) + e, lo, hi);
                            }
                        }
                    }
                    if (live) p.part_lse[prow] = m + log2f(l);
                }
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool BF16, bool FP8>
static cudaError_t prepare_wide_k() {
    using C = WideCfg<D>;
    static_assert(sizeof(WideBarriers) <= 512, "barrier block");
    if constexpr (FP8) {
        // the register split (setmaxnreg) draws on the launch's registers: a build that runs the kernel at
        // another per-thread count would leave the softmax warps waiting for registers, so it is refused
        static const cudaError_t regs = [] {
            cudaFuncAttributes fa{};
            const cudaError_t r = cudaFuncGetAttributes(&fa, prefix_wide_kernel<D, BF16, FP8>);
            if (r != cudaSuccess) return r;
            return fa.numRegs == C::REGS_LAUNCH_E4M3 ? cudaSuccess : cudaErrorInvalidConfiguration;
        }();
        if (regs != cudaSuccess) return regs;
    }
    cudaError_t e =
        cudaFuncSetAttribute(prefix_wide_kernel<D, BF16, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(prefix_wide_kernel<D, BF16, FP8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

template <int D, bool FP8>
static cudaError_t prepare_wide_d(bool bf16) {
    return bf16 ? prepare_wide_k<D, true, FP8>() : prepare_wide_k<D, false, FP8>();
}

cudaError_t prepare_wide(int head_dim, bool bf16, bool fp8) {
    switch (head_dim) {
        case 64: return fp8 ? prepare_wide_d<64, true>(bf16) : prepare_wide_d<64, false>(bf16);
        case 128: return fp8 ? prepare_wide_d<128, true>(bf16) : prepare_wide_d<128, false>(bf16);
        default: return cudaErrorInvalidValue;
    }
}

template <int D, bool BF16, bool FP8>
static void launch_wide_k(int ctas, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const PrefixParams& p, cudaStream_t stream) {
    constexpr int threads = FP8 ? WideCfg<D>::THREADS_E4M3 : WideCfg<D>::THREADS;
    prefix_wide_kernel<D, BF16, FP8><<<ctas, threads, WideCfg<D>::SMEM, stream>>>(tq, tk, tv, p);
}

template <int D>
static void launch_wide_d(bool bf16, bool fp8, int ctas, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const PrefixParams& p, cudaStream_t stream) {
    if (bf16) {
        if (fp8) launch_wide_k<D, true, true>(ctas, tq, tk, tv, p, stream);
        else launch_wide_k<D, true, false>(ctas, tq, tk, tv, p, stream);
    } else {
        if (fp8) launch_wide_k<D, false, true>(ctas, tq, tk, tv, p, stream);
        else launch_wide_k<D, false, false>(ctas, tq, tk, tv, p, stream);
    }
}

cudaError_t launch_wide(int head_dim, bool bf16, int ctas, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const PrefixParams& p, cudaStream_t stream, bool fp8) {
    if (ctas == 0 || p.num_units == 0) return cudaSuccess;
    if (p.bq <= 0 || p.bq * p.G > 32) return cudaErrorInvalidValue;
    switch (head_dim) {
        case 64: launch_wide_d<64>(bf16, fp8, ctas, tq, tk, tv, p, stream); break;
        case 128: launch_wide_d<128>(bf16, fp8, ctas, tq, tk, tv, p, stream); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace bsp
