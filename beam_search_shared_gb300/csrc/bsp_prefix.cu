// Prompt (prefix) attention of the cascade on 5th-generation tensor cores
// (TensorRT-LLM PR #21738, "Add opt-in cascade attention for wide beam search
// on KVCM V2", description: "Prefix: the shared prompt is attended once per
// request"; all beam_width x GQA-group query rows of a request share one K/V
// stream, which makes Q*K^T and P*V dense contractions).
//
// One CTA = one work unit: (request b, kv head g, query-row block, range of
// 64-key tiles). Query rows of the block are (beam w, head j) pairs, row
// = w_local * G + j, at most 128 (the MMA M). Only the valid prompt rows
// [0, P_b) are read (TensorRT-Model-Connect PR #2202, "prefill and decode
// over the cached prefix, not the whole KV allocation").
//
// Warp roles (192 threads):
//   warp 0     TMA producer: Q once, then K and V tiles of the unit's pages
//              (beam 0's prompt pages) into a STAGES-deep ring;
//   warp 1     TMEM allocation and the MMA issuer (one thread):
//              S[i%2] = Q K_i^T, then O += P_{i-1} V_{i-1};
//   warps 2-5  softmax: thread <-> query row <-> TMEM lane; reads S from
//              TMEM, online softmax in base 2 with a lazy rescale of O (only
//              when the row maximum grows by more than 2^8), writes P (16-bit,
//              swizzled K-major) to shared memory, epilogue writes the
//              normalised partial O and its log2-sum-exp2 (fp32) to the
//              workspace for the tail kernel's merge.
// TMEM columns: S0 [0,64), S1 [64,128), O [128, 128+D).
// Every wait is bounded (2 s per CTA); on expiry the CTA flags
// BSP_DEVFLAG_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "bsp_internal.h"
#include "bsp_ptx.cuh"
#include "../../include/bsp.h"

namespace bsp {

template <int D>
struct PrefixCfg {
    static constexpr int TK = kTileKeys;
    static constexpr int NC = D / 64;                       // 128-byte column regions per row
    static constexpr int STAGES = D == 64 ? 6 : (D == 128 ? 4 : 2);
    static constexpr int Q_BYTES = kRowsPerBlock * D * 2;   // NC regions of 128 rows x 128 B
    static constexpr int P_BYTES = kRowsPerBlock * TK * 2;  // one region
    static constexpr int KV_BYTES = TK * D * 2;             // one of K or V per stage
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int OFF_P = Q_BYTES;
    static constexpr int OFF_STAGE = Q_BYTES + P_BYTES;
    static constexpr int OFF_BAR = OFF_STAGE + STAGES * STAGE_BYTES;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;       // barriers + alignment slack
    static constexpr int S_COL = 0;
    static constexpr int O_COL = 2 * TK;
    static constexpr uint32_t TMEM_COLS = (O_COL + D) <= 256 ? 256u : 512u;
    static constexpr int THREADS = 192;
};

struct PrefixBarriers {
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t q_full;
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full;
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
prefix_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefixParams p) {
    using C = PrefixCfg<D>;
    constexpr int TK = C::TK, NC = C::NC, STAGES = C::STAGES;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sP = smem + C::OFF_P;
    PrefixBarriers* bars = reinterpret_cast<PrefixBarriers*>(smem + C::OFF_BAR);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint64_t deadline = globaltimer_ns() + 2000000000ull;

    // ---- unit
    const int* u = p.units + static_cast<long long>(blockIdx.x) * kUnitFields;
    const int b = __ldg(u + kUnitReq), g = __ldg(u + kUnitKvHead), rb = __ldg(u + kUnitRowBlock);
    const int kt0 = __ldg(u + kUnitTile0), kt1 = __ldg(u + kUnitTile1), part = __ldg(u + kUnitPart);
    const int* rq = p.req + b * kReqFields;
    const int P = __ldg(rq + kReqPrefix);
    const int page_off = __ldg(rq + kReqPageOff);
    const int key_begin = kt0 * TK;
    const int key_end = min(kt1 * TK, P);
    const int ntiles = kt1 - kt0;
    const int w0 = rb * p.Wblk;
    const int nbeams = min(p.Wblk, p.W - w0);
    const int M = nbeams * p.G;

    // ---- setup
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        mbar_init(&bars->q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_free[i], 128);
        }
        mbar_init(&bars->p_full, 128);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 1) tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
    // zero the query rows the TMA box does not cover, so padded rows stay finite
    {
        const int filled = p.Wblk * p.G;
        const int nz = (kRowsPerBlock - filled) * 8;  // 16-byte chunks per region
        for (int c = 0; c < NC; ++c)
            for (int idx = tid; idx < nz; idx += C::THREADS)
                reinterpret_cast<uint4*>(sQ + c * kRowsPerBlock * 128 + filled * 128)[idx] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ================= TMA producer =================
        const int* pg = p.pages + page_off;
        const int npages = (P + (1 << p.ps_log2) - 1) >> p.ps_log2;
        const int ps = 1 << p.ps_log2;
        const int BR = ps < TK ? ps : TK;  // rows per box
        int win_base = -1, my_page = 0;
        int issued = 0;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars->q_full, NC * p.Wblk * p.G * 128);
            for (int c = 0; c < NC; ++c)
                tma_load_3d(sQ + c * kRowsPerBlock * 128, &tm_q, &bars->q_full, c * 64, g * p.G, b * p.W + w0);
        }
        bool ok = true;
        for (int i = 0; i < ntiles && ok; ++i) {
            const int s = i % STAGES;
            if (i >= STAGES) {
                ok = mbar_wait(&bars->kv_empty[s], ((i / STAGES) - 1) & 1, abort_flag, deadline);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
            }
            const int key0 = key_begin + i * TK;
            const int valid = min(TK, key_end - key0);
            const int nchunks = (valid + BR - 1) / BR;
            uint8_t* sK = smem + C::OFF_STAGE + s * C::STAGE_BYTES;
            uint8_t* sV = sK + C::KV_BYTES;
            if (lane == 0) mbar_arrive_expect_tx(&bars->kv_full[s], nchunks * BR * 128 * NC * 2);
            for (int ch = 0; ch < nchunks; ++ch) {
                const int key = key0 + ch * BR;
                const int pidx = key >> p.ps_log2;
                if (win_base < 0 || pidx >= win_base + 32) {  // warp-uniform
                    win_base = pidx;
                    my_page = (win_base + lane < npages) ? __ldg(pg + win_base + lane) : 0;
                }
                int page = __shfl_sync(FULL, my_page, pidx - win_base);
                if (static_cast<unsigned>(page) >= static_cast<unsigned>(p.num_pages)) {
                    if (lane == 0) atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
                    page = 0;
                }
                const int row = ((page * p.Hkv + g) << p.ps_log2) + (key & (ps - 1));
                if (lane == 0) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        tma_load_2d(sK + c * TK * 128 + ch * BR * 128, &tm_k, &bars->kv_full[s], c * 64, row);
                        tma_load_2d(sV + c * TK * 128 + ch * BR * 128, &tm_v, &bars->kv_full[s], c * 64, row);
                    }
                }
            }
            issued = i + 1;
        }
        if (!ok) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
            }
            // drain: let this CTA's own copies land before the CTA exits
            const uint64_t dl = globaltimer_ns() + 200000000ull;
            for (int j = max(0, issued - STAGES); j < issued; ++j)
                while (!mbar_try_wait(&bars->kv_full[j % STAGES], (j / STAGES) & 1) && globaltimer_ns() < dl) {
                }
            if (lane == 0) {
                while (!mbar_try_wait(&bars->q_full, 0) && globaltimer_ns() < dl) {
                }
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t ID_QK = idesc_f16(128, TK, BF16, false);
            constexpr uint32_t ID_PV = idesc_f16(128, D, BF16, true);
            const uint32_t q_addr = smem_u32(sQ);
            const uint32_t p_addr = smem_u32(sP);
            bool ok = mbar_wait(&bars->q_full, 0, abort_flag, deadline);
            int pv_issued = 0;
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait(&bars->p_full, j & 1, abort_flag, deadline)) return false;
                tc_fence_after();
                const int sj = j % STAGES;
                const uint32_t v_addr = smem_u32(smem + C::OFF_STAGE + sj * C::STAGE_BYTES + C::KV_BYTES);
#pragma unroll
                for (int kk = 0; kk < TK / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(p_addr + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(v_addr + kk * 16 * 128, TK * 128, 1024);
                    mma_f16(tmem + C::O_COL, a, bd, ID_PV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars->o_done);
                mma_commit(&bars->kv_empty[sj]);
                pv_issued = j + 1;
                return true;
            };
            for (int i = 0; i < ntiles && ok; ++i) {
                const int s = i % STAGES;
                ok = mbar_wait(&bars->kv_full[s], (i / STAGES) & 1, abort_flag, deadline);
                if (ok && i >= 2) ok = mbar_wait(&bars->s_free[i & 1], ((i - 2) >> 1) & 1, abort_flag, deadline);
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_addr = smem_u32(smem + C::OFF_STAGE + s * C::STAGE_BYTES);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(q_addr + (kk >> 2) * (kRowsPerBlock * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(k_addr + (kk >> 2) * (TK * 128) + (kk & 3) * 32, 16, 1024);
                    mma_f16(tmem + C::S_COL + (i & 1) * TK, a, bd, ID_QK, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars->s_full[i & 1]);
                if (i >= 1) ok = issue_pv(i - 1);
            }
            if (ok && ntiles > 0) ok = issue_pv(ntiles - 1);
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
            }
            (void)pv_issued;
            // drain: every MMA issued by this thread completes before TMEM is freed
            mma_commit(&bars->drain);
            const uint64_t dl = globaltimer_ns() + 200000000ull;
            while (!mbar_try_wait(&bars->drain, 0) && globaltimer_ns() < dl) {
            }
        }
    } else {
        // ================= softmax warps =================
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float sl2 = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int key0 = key_begin + i * TK;
            const int valid = min(TK, key_end - key0);
            ok = mbar_wait(&bars->s_full[i & 1], (i >> 1) & 1, abort_flag, deadline);
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[2][32];
            tmem_ld32(lane_base + C::S_COL + (i & 1) * TK, sr[0]);
            tmem_ld32(lane_base + C::S_COL + (i & 1) * TK + 32, sr[1]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bars->s_free[i & 1]);
            float sv[TK];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < TK; ++c) {
                const float v = (c < valid) ? __uint_as_float(sr[c >> 5][c & 31]) * sl2 : -INFINITY;
                sv[c] = v;
                mx = fmaxf(mx, v);
            }
            if (i > 0) {
                // P_{i-1} V_{i-1} has finished: O may be rescaled and the P buffer reused
                ok = mbar_wait(&bars->o_done, (i - 1) & 1, abort_flag, deadline);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                tc_fence_after();
                const bool need = mx > m + 8.0f;
                if (__any_sync(FULL, need)) {
                    const float alpha = need ? exp2f(m - mx) : 1.0f;
                    if (need) {
                        m = mx;
                        l *= alpha;
                    }
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t orr[32];
                        tmem_ld32(lane_base + C::O_COL + c0, orr);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(lane_base + C::O_COL + c0, orr);
                    }
                    tmem_wait_st();
                }
            } else {
                m = mx;
            }
            // probabilities, row sum, P to shared memory (128-byte swizzle, K-major)
            float rs = 0.f;
            uint32_t pk[TK / 2];
#pragma unroll
            for (int c = 0; c < TK; c += 2) {
                const float p0 = exp2f(sv[c] - m);
                const float p1 = exp2f(sv[c + 1] - m);
                rs += p0 + p1;
                pk[c >> 1] = pack2<BF16>(p0, p1);
            }
            l += rs;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
                *reinterpret_cast<uint4*>(sP + row * 128 + ((cc ^ (row & 7)) << 4)) =
                    make_uint4(pk[cc * 4], pk[cc * 4 + 1], pk[cc * 4 + 2], pk[cc * 4 + 3]);
            if (valid < TK) {
                // last tile: zero V rows past the valid keys (stale or garbage rows times P = 0
                // must not produce NaN)
                const int s = i % STAGES;
                ok = mbar_wait(&bars->kv_full[s], (i / STAGES) & 1, abort_flag, deadline);
                ok = __all_sync(FULL, ok);
                if (!ok) break;
                uint8_t* sV = smem + C::OFF_STAGE + s * C::STAGE_BYTES + C::KV_BYTES;
                const int nzc = (TK - valid) * 8;  // 16-byte chunks per region
                const int t = tid - 64;
                for (int c = 0; c < NC; ++c)
                    for (int idx = t; idx < nzc; idx += 128)
                        reinterpret_cast<uint4*>(sV + c * TK * 128 + valid * 128)[idx] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->p_full);
        }
        if (ok && ntiles > 0) {
            ok = mbar_wait(&bars->o_done, (ntiles - 1) & 1, abort_flag, deadline);
            ok = __all_sync(FULL, ok);
        }
        if (ok && ntiles > 0) {
            tc_fence_after();
            const bool live = row < M;
            const int wl = row / p.G, jh = row % p.G;
            const long long prow = (static_cast<long long>(part) * p.W + (w0 + wl)) * p.Hq + g * p.G + jh;
            float4* dst = reinterpret_cast<float4*>(p.part_o + prow * D);
            const float inv = 1.0f / l;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t orr[32];
                tmem_ld32(lane_base + C::O_COL + c0, orr);
                tmem_wait_ld();
                if (live) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[(c0 >> 2) + e] = make_float4(__uint_as_float(orr[4 * e]) * inv, __uint_as_float(orr[4 * e + 1]) * inv,
                                                         __uint_as_float(orr[4 * e + 2]) * inv, __uint_as_float(orr[4 * e + 3]) * inv);
                }
            }
            if (live) p.part_lse[prow] = m + log2f(l);
        }
        if (!ok) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicOr(p.status, BSP_DEVFLAG_TIMEOUT);
            }
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

template <int D, bool BF16>
static cudaError_t launch_prefix_t(int num_units, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const PrefixParams& p, cudaStream_t stream) {
    using C = PrefixCfg<D>;
    static_assert(sizeof(PrefixBarriers) <= 256, "barrier block");
    cudaError_t e = cudaFuncSetAttribute(prefix_attn_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    prefix_attn_kernel<D, BF16><<<num_units, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

cudaError_t launch_prefix(int head_dim, bool bf16, int num_units, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const PrefixParams& p, cudaStream_t stream) {
    if (num_units == 0) return cudaSuccess;
    switch (head_dim) {
        case 64: return bf16 ? launch_prefix_t<64, true>(num_units, tq, tk, tv, p, stream)
                             : launch_prefix_t<64, false>(num_units, tq, tk, tv, p, stream);
        case 128: return bf16 ? launch_prefix_t<128, true>(num_units, tq, tk, tv, p, stream)
                              : launch_prefix_t<128, false>(num_units, tq, tk, tv, p, stream);
        case 256: return bf16 ? launch_prefix_t<256, true>(num_units, tq, tk, tv, p, stream)
                              : launch_prefix_t<256, false>(num_units, tq, tk, tv, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bsp
