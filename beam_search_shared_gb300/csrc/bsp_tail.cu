// Tail attention with the log-sum-exp merge fused into its epilogue
// (TensorRT-LLM PR #21738, "Add opt-in cascade attention for wide beam search
// on KVCM V2": description, the tail half of the cascade: the tokens a beam
// generated itself, found through cache_indirection; the commit that fuses the
// tail runs its attention and the join with the prompt part in a single launch per layer).
//
// One CTA per beam row r = b*W + w (per row and head pass when the step has
// fewer rows than SMs). The row's tail positions j = P_b + t
// (t < T_b <= 8) are resolved once: threads t look up the source beam
// cache_indirection[b][w][j] and that beam's page id, and leave the row's
// physical offset in shared memory. The warps then serve the query heads: a
// head's row of head_dim 16-bit elements is read by D/8 lanes with 16-byte
// loads (32/(D/8) heads per warp pass), every K and V chunk of the head's tail
// rows is issued at once, and the softmax over those rows is merged with the
// request's prompt partial states (one per key split) by log-sum-exp: the
// head's lanes load the partial LSEs in parallel and reduce their maximum by
// shuffles, then the partial O rows arrive a few splits per round. O is
// written in the q dtype and LSE in fp32. So one chain of dependent lookups
// serves all Hq heads of the row. All softmax arithmetic is in base 2 on
// scores pre-scaled by softmax_scale * log2(e).
//
// A prefill request whose cached keys the plan split is merged here too: its
// prompt tokens are the rows (w < the request's rows, W the longest prompt of
// the batch; q, O and LSE at the request's first row + w), with no tail keys.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "bsp_internal.h"
#include "bsp_prompt.cuh"
#include "bsp_ptx.cuh"
#include "../../include/bsp.h"

namespace bsp {

namespace {

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
            float2 v = __bfloat1622float2(h);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        } else {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 v = __half22float2(h);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
}

// 8 E4M3 codes as fp32, exactly (through binary16)
__device__ __forceinline__ void unpack8_e4m3(const uint2& u, float (&f)[8]) {
    const uint4 h = e4m3x8_to_16<false>(u);
    const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

template <bool BF16>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        } else {
            __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

constexpr int kTailThreads = 128;

// MAXT: tail rows held in registers, the batch's longest tail rounded up to 2, 4 or 8.
// MAXP: head passes whose tail state is held in registers across the wait for the prompt kernel
// (passes = Hq / (4 warps x heads per warp pass), rounded up to 1, 2 or 4; more passes are done
// in groups of MAXP).
// FP8: E4M3 pools (a lane reads 8 one-byte codes of a row instead of 8 16-bit elements; the keys'
// scale is folded into scale_log2, the values' scale into the tail's share of O).
template <int D, bool BF16, int MAXT, int MAXP, bool FP8>
__global__ void __launch_bounds__(kTailThreads) tail_merge_kernel(TailParams p) {
    constexpr int LPR = D / 8;       // lanes per K/V row
    constexpr int HPW = 32 / LPR;    // heads per warp pass
    constexpr int NW = kTailThreads / 32;
    constexpr unsigned FULL = 0xffffffffu;
    __shared__ long long s_off[BSP_MAX_TAIL];  // element offset of tail row t for kv head 0, -1 if unreadable

    if (p.graph_hdr != nullptr) {
        // a launch replayed from a CUDA graph: the plan staged since must have the captured shape
        const int4 h0 = __ldg(reinterpret_cast<const int4*>(p.graph_hdr));
        const int4 h1 = __ldg(reinterpret_cast<const int4*>(p.graph_hdr) + 1);
        if (h0.z != p.B || h1.x != p.W || h1.z != 0 || h1.w > p.graph_max_tail) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.status, BSP_DEVFLAG_GRAPH);
            return;
        }
    }
    const int r = blockIdx.x;
    const int b = r / p.W;
    const int w = r % p.W;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int4 rq = __ldg(reinterpret_cast<const int4*>(p.req + b * kReqFields));
    const int P = rq.x, T = rq.y, nsplit = rq.z, part_off = rq.w;
    if (__ldg(p.req + b * kReqFields + kReqFused)) return;  // the prompt kernel finished this request
    // the request's rows (beams; prompt tokens of a prefill, W = the longest prompt) and its first row
    const int4 rq3 = __ldg(reinterpret_cast<const int4*>(p.req + b * kReqFields + 8));
    if (w >= rq3.x) return;                                  // kReqRows
    const long long orow = static_cast<long long>(rq3.z) + w;  // kReqRowOff: the row of q, o and lse

    // ---- resolve the row's tail positions once (source beam, page, slot)
    if (tid < T) {
        const int pos = P + tid;
        const int src = __ldg(p.ci + (static_cast<long long>(b) * p.W + w) * p.max_seq + pos);
        long long off = -1;
        if (static_cast<unsigned>(src) < static_cast<unsigned>(p.W)) {
            const int page = __ldg(p.beam_pages + (static_cast<long long>(b) * p.W + src) * p.beam_pages_stride +
                                   (pos >> p.ps_log2));
            if (static_cast<unsigned>(page) < static_cast<unsigned>(p.num_pages))
                off = ((static_cast<long long>(page) * p.Hkv << p.ps_log2) + (pos & ((1 << p.ps_log2) - 1))) * D;
        }
        if (off < 0) atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
        s_off[tid] = off;
    }
    __syncthreads();

    const int hs = lane / LPR;  // head slot within the warp pass
    const int li = lane % LPR;  // 16-byte chunk of the row
    const long long head_stride = static_cast<long long>(D) << p.ps_log2;  // next kv head, same page/slot
    const long long pstride = static_cast<long long>(p.W) * p.Hq;          // rows of one partial slot
    const int passes = (p.Hq + NW * HPW - 1) / (NW * HPW);

    // with few rows the head passes are spread over gridDim.y CTAs per row
    for (int pg = blockIdx.y * MAXP; pg < passes; pg += gridDim.y * MAXP) {
        // ---- the tail keys of this group of head passes: softmax state (m, l) and the lane's
        // 8 columns of sum_t 2^(s_t - m) V_t. Everything read here was written before the prompt
        // kernel started, so a CTA launched as a dependent of the prompt kernel computes it while
        // that kernel still runs.
        float tm[MAXP], tl[MAXP], acc[MAXP][8];
#pragma unroll
        for (int pi = 0; pi < MAXP; ++pi) {
            const int h = (pg + pi) * NW * HPW + warp * HPW + hs;
            const bool active = pg + pi < passes && h < p.Hq;  // lanes of a head slot agree
            const int hh = active ? h : 0;
            const int g = hh / p.G;
            const uint4 qraw = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                                     (orow * p.Hq + hh) * D) +
                                     li);
            // a lane's 8 elements of a K or V row: 16 bytes, or 8 E4M3 codes (the upper half unused)
            uint4 kraw[MAXT], vraw[MAXT];
            bool ok[MAXT];
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                const long long off = t < T ? s_off[t] : -1;
                ok[t] = active && off >= 0;
                kraw[t] = vraw[t] = make_uint4(0, 0, 0, 0);
                if (ok[t]) {
                    const long long e = off + g * head_stride;  // element offset
                    if constexpr (FP8) {
                        const uint2 kk = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.k_pool) + e) + li);
                        const uint2 vv = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.v_pool) + e) + li);
                        kraw[t] = make_uint4(kk.x, kk.y, 0, 0);
                        vraw[t] = make_uint4(vv.x, vv.y, 0, 0);
                    } else {
                        kraw[t] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_pool) + e) + li);
                        vraw[t] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v_pool) + e) + li);
                    }
                }
            }
            float q[8];
            unpack8<BF16>(qraw, q);
            float sc[MAXT];
            float m = -INFINITY;
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                sc[t] = -INFINITY;
                if (t < T) {  // block-uniform: rows past the request's tail cost nothing
                    float kf[8];
                    if constexpr (FP8) unpack8_e4m3(make_uint2(kraw[t].x, kraw[t].y), kf);
                    else unpack8<BF16>(kraw[t], kf);
                    float dot = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) dot = fmaf(q[e], kf[e], dot);
#pragma unroll
                    for (int off = LPR / 2; off >= 1; off >>= 1) dot += __shfl_xor_sync(FULL, dot, off);
                    if (ok[t]) sc[t] = dot * p.scale_log2;
                    m = fmaxf(m, sc[t]);
                }
            }
            float l = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[pi][e] = 0.f;
            if (m != -INFINITY) {
#pragma unroll
                for (int t = 0; t < MAXT; ++t) {
                    if (!ok[t]) continue;
                    const float e_s = exp2f(sc[t] - m);
                    float vf[8];
                    if constexpr (FP8) unpack8_e4m3(make_uint2(vraw[t].x, vraw[t].y), vf);
                    else unpack8<BF16>(vraw[t], vf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[pi][e] = fmaf(e_s, vf[e], acc[pi][e]);
                    l += e_s;
                }
            }
            tm[pi] = m;
            tl[pi] = l;
        }

        // ---- wait for the prompt kernel's partial states (returns at once when launched plainly)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // the partial states are read coherently below (never through the read-only path, whose
        // loads the compiler may move above the wait)

        // ---- merge with the prompt partial states by log-sum-exp (base 2). Split 0 of every head
        // of the group is loaded in one round; with more splits, the lanes of a head slot load the
        // other partial LSEs in parallel (lane li: splits 1 + li, 1 + li + LPR, ...) and reduce
        // their maximum by shuffles, then the other partial O rows arrive KB splits per round.
        constexpr int KMAX = (kExtraParts + LPR - 1) / LPR;  // unrolled loads: up to kExtraParts more splits
        constexpr int KB = 4;
        float lse0[MAXP];
        float4 o0a[MAXP], o0b[MAXP];
#pragma unroll
        for (int pi = 0; pi < MAXP; ++pi) {
            const int h = (pg + pi) * NW * HPW + warp * HPW + hs;
            const bool active = pg + pi < passes && h < p.Hq;
            lse0[pi] = -INFINITY;
            o0a[pi] = o0b[pi] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (active && nsplit > 0) {
                const long long prow = (static_cast<long long>(part_off) * p.W + w) * p.Hq + h;
                lse0[pi] = ld_dep(p.part_lse + prow);
                const float4* po = reinterpret_cast<const float4*>(p.part_o + prow * D) + li * 2;
                o0a[pi] = ld_dep(po);
                o0b[pi] = ld_dep(po + 1);
            }
        }
#pragma unroll
        for (int pi = 0; pi < MAXP; ++pi) {
            const int h = (pg + pi) * NW * HPW + warp * HPW + hs;
            const bool active = pg + pi < passes && h < p.Hq;  // every lane still takes part in the shuffles
            const long long prow = (static_cast<long long>(part_off) * p.W + w) * p.Hq + (active ? h : 0);
            const float m = tm[pi], l = tl[pi];
            float Lmax = (l > 0.f) ? m + log2f(l) : -INFINITY;
            Lmax = fmaxf(Lmax, lse0[pi]);
            if (nsplit > 1) {  // block-uniform
                float lsev[KMAX];
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    const int sp = 1 + k * LPR + li;
                    lsev[k] = (active && sp < nsplit) ? ld_dep(p.part_lse + prow + sp * pstride) : -INFINITY;
                }
#pragma unroll
                for (int k = 0; k < KMAX; ++k) Lmax = fmaxf(Lmax, lsev[k]);
                // a request may hold more splits when others of the batch have none (the planner's bound
                // is batch + kExtraParts in all): the rest, one load per lane at a time
                for (int sp = 1 + KMAX * LPR + li; active && sp < nsplit; sp += LPR)
                    Lmax = fmaxf(Lmax, ld_dep(p.part_lse + prow + sp * pstride));
#pragma unroll
                for (int off = LPR / 2; off >= 1; off >>= 1) Lmax = fmaxf(Lmax, __shfl_xor_sync(FULL, Lmax, off));
            }
            float out[8];
            float lse2;
            if (Lmax == -INFINITY) {
#pragma unroll
                for (int e = 0; e < 8; ++e) out[e] = 0.f;
                lse2 = -INFINITY;
            } else {
                // tail weight exp2(m + log2 l - Lmax) times O_t = acc / l, then split 0
                const float ft = (l > 0.f) ? exp2f(m - Lmax) : 0.f;
                const float fv = ft * p.v_scale;          // the tail's values in their E4M3 scale (1 otherwise)
                const float w0 = exp2f(lse0[pi] - Lmax);  // 0 without a prompt
                float sum = l * ft + w0;
                out[0] = fmaf(w0, o0a[pi].x, acc[pi][0] * fv);
                out[1] = fmaf(w0, o0a[pi].y, acc[pi][1] * fv);
                out[2] = fmaf(w0, o0a[pi].z, acc[pi][2] * fv);
                out[3] = fmaf(w0, o0a[pi].w, acc[pi][3] * fv);
                out[4] = fmaf(w0, o0b[pi].x, acc[pi][4] * fv);
                out[5] = fmaf(w0, o0b[pi].y, acc[pi][5] * fv);
                out[6] = fmaf(w0, o0b[pi].z, acc[pi][6] * fv);
                out[7] = fmaf(w0, o0b[pi].w, acc[pi][7] * fv);
                for (int sp0 = 1; sp0 < nsplit; sp0 += KB) {
                    float ls[KB];
                    float4 a0[KB], a1[KB];
#pragma unroll
                    for (int u = 0; u < KB; ++u) {
                        const int sp = sp0 + u;
                        ls[u] = -INFINITY;
                        a0[u] = a1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (active && sp < nsplit) {
                            ls[u] = ld_dep(p.part_lse + prow + sp * pstride);
                            const float4* po = reinterpret_cast<const float4*>(p.part_o + (prow + sp * pstride) * D) + li * 2;
                            a0[u] = ld_dep(po);
                            a1[u] = ld_dep(po + 1);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < KB; ++u) {
                        const float wgt = exp2f(ls[u] - Lmax);  // 0 for splits past nsplit
                        out[0] = fmaf(wgt, a0[u].x, out[0]);
                        out[1] = fmaf(wgt, a0[u].y, out[1]);
                        out[2] = fmaf(wgt, a0[u].z, out[2]);
                        out[3] = fmaf(wgt, a0[u].w, out[3]);
                        out[4] = fmaf(wgt, a1[u].x, out[4]);
                        out[5] = fmaf(wgt, a1[u].y, out[5]);
                        out[6] = fmaf(wgt, a1[u].z, out[6]);
                        out[7] = fmaf(wgt, a1[u].w, out[7]);
                        sum += wgt;
                    }
                }
                const float inv = 1.f / sum;
#pragma unroll
                for (int e = 0; e < 8; ++e) out[e] *= inv;
                lse2 = Lmax + log2f(sum);
            }
            if (!active) continue;
            uint16_t* obase = static_cast<uint16_t*>(p.o) + (orow * p.Hq + h) * D;
            reinterpret_cast<uint4*>(obase)[li] = pack8<BF16>(out);
            if (li == 0) p.lse[orow * p.Hq + h] = p.lse_base2 ? lse2 : lse2 * 0.69314718055994530942f;
        }
    }
}

template <int D, bool BF16, int MAXT, int MAXP, bool FP8>
static cudaError_t launch_tail_k(const TailParams& p, bool after_prefix, int pass_ctas, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.B) * p.W;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows), static_cast<unsigned>(pass_ctas));
    cfg.blockDim = dim3(kTailThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_prefix ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, tail_merge_kernel<D, BF16, MAXT, MAXP, FP8>, p);
}

// head passes of a 128-thread CTA: Hq / (4 warps x heads per warp pass)
template <int D>
static int tail_passes(int Hq) {
    constexpr int hpw = 32 / (D / 8);
    return (Hq + 4 * hpw - 1) / (4 * hpw);
}

// SMs of the current device (cached per device)
static int device_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

template <int D, bool BF16, int MAXT, bool FP8>
static cudaError_t launch_tail_p(const TailParams& p, bool after_prefix, cudaStream_t stream) {
    const int passes = tail_passes<D>(p.Hq);
    const long long rows = static_cast<long long>(p.B) * p.W;
    // fewer rows than SMs: one CTA per (row, head pass), so a row's heads merge in parallel
    if (passes > 1 && rows < device_sms()) return launch_tail_k<D, BF16, MAXT, 1, FP8>(p, after_prefix, passes, stream);
    if (passes <= 1) return launch_tail_k<D, BF16, MAXT, 1, FP8>(p, after_prefix, 1, stream);
    if (passes <= 2) return launch_tail_k<D, BF16, MAXT, 2, FP8>(p, after_prefix, 1, stream);
    return launch_tail_k<D, BF16, MAXT, 4, FP8>(p, after_prefix, 1, stream);
}

template <int D, bool BF16, bool FP8>
static cudaError_t launch_tail_t(const TailParams& p, int max_tail_len, bool after_prefix, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.B) * p.W;
    if (rows == 0) return cudaSuccess;
    if (max_tail_len <= 2) return launch_tail_p<D, BF16, 2, FP8>(p, after_prefix, stream);
    if (max_tail_len <= 4) return launch_tail_p<D, BF16, 4, FP8>(p, after_prefix, stream);
    return launch_tail_p<D, BF16, 8, FP8>(p, after_prefix, stream);
}

// the same L1/shared split as the prompt kernel, so SMs are not reconfigured between the
// kernels of a step
template <int D, bool BF16, int MAXT, bool FP8>
static cudaError_t prepare_tail_p(int Hq) {
    const cudaFuncAttribute a = cudaFuncAttributePreferredSharedMemoryCarveout;
    const int passes = tail_passes<D>(Hq);
    // the one-pass variant also serves steps with fewer rows than SMs
    const cudaError_t e =
        cudaFuncSetAttribute(tail_merge_kernel<D, BF16, MAXT, 1, FP8>, a, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess || passes <= 1) return e;
    if (passes <= 2) return cudaFuncSetAttribute(tail_merge_kernel<D, BF16, MAXT, 2, FP8>, a, cudaSharedmemCarveoutMaxShared);
    return cudaFuncSetAttribute(tail_merge_kernel<D, BF16, MAXT, 4, FP8>, a, cudaSharedmemCarveoutMaxShared);
}

template <int D, bool BF16, bool FP8>
static cudaError_t prepare_tail_t(int max_tail_len, int Hq) {
    if (max_tail_len <= 2) return prepare_tail_p<D, BF16, 2, FP8>(Hq);
    if (max_tail_len <= 4) return prepare_tail_p<D, BF16, 4, FP8>(Hq);
    return prepare_tail_p<D, BF16, 8, FP8>(Hq);
}

template <int D, bool FP8>
static cudaError_t prepare_tail_d(bool bf16, int max_tail_len, int Hq) {
    return bf16 ? prepare_tail_t<D, true, FP8>(max_tail_len, Hq) : prepare_tail_t<D, false, FP8>(max_tail_len, Hq);
}

template <int D, bool FP8>
static cudaError_t launch_tail_d(bool bf16, int max_tail_len, const TailParams& p, bool after_prefix,
                                 cudaStream_t stream) {
    return bf16 ? launch_tail_t<D, true, FP8>(p, max_tail_len, after_prefix, stream)
                : launch_tail_t<D, false, FP8>(p, max_tail_len, after_prefix, stream);
}

// E4M3 pools at head_dim 64 and 128 only
cudaError_t prepare_tail(int head_dim, bool bf16, int max_tail_len, int num_q_heads, bool fp8) {
    switch (head_dim) {
        case 64: return fp8 ? prepare_tail_d<64, true>(bf16, max_tail_len, num_q_heads)
                            : prepare_tail_d<64, false>(bf16, max_tail_len, num_q_heads);
        case 128: return fp8 ? prepare_tail_d<128, true>(bf16, max_tail_len, num_q_heads)
                             : prepare_tail_d<128, false>(bf16, max_tail_len, num_q_heads);
        case 256: return fp8 ? cudaErrorInvalidValue : prepare_tail_d<256, false>(bf16, max_tail_len, num_q_heads);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tail(int head_dim, bool bf16, int max_tail_len, const TailParams& p, bool after_prefix,
                        cudaStream_t stream, bool fp8) {
    switch (head_dim) {
        case 64: return fp8 ? launch_tail_d<64, true>(bf16, max_tail_len, p, after_prefix, stream)
                            : launch_tail_d<64, false>(bf16, max_tail_len, p, after_prefix, stream);
        case 128: return fp8 ? launch_tail_d<128, true>(bf16, max_tail_len, p, after_prefix, stream)
                             : launch_tail_d<128, false>(bf16, max_tail_len, p, after_prefix, stream);
        case 256: return fp8 ? cudaErrorInvalidValue
                             : launch_tail_d<256, false>(bf16, max_tail_len, p, after_prefix, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bsp
