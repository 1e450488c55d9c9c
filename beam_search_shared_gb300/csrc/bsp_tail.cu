// Tail attention with the log-sum-exp merge fused into its epilogue
// (TensorRT-LLM PR #21738, "Add opt-in cascade attention for wide beam search
// on KVCM V2": description, "Tail: each beam's own generated tokens, gathered
// through cache_indirection"; the tail and the merge with the prefix result
// run as one launch per layer, commit "...fused tail, sized workspace").
//
// One warp per (beam row r, query head h). A row of head_dim 16-bit elements
// is read by D/8 lanes with 16-byte loads, so a warp walks 32/(D/8) tail rows
// at once. Tail position j = P_b + t of beam w is read from the page table of
// beam cache_indirection[b][w][j]. The warp keeps an online softmax over its
// <= 8 rows, combines its row groups by shuffles, then merges the tail state
// with the request's prompt partial states (one per key split) by
// log-sum-exp and writes O (q dtype) and LSE (fp32). All softmax arithmetic is
// in base 2 on scores pre-scaled by softmax_scale * log2(e).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "bsp_internal.h"
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

template <int D, bool BF16>
__global__ void __launch_bounds__(128) tail_merge_kernel(TailParams p) {
    constexpr int LPR = D / 8;     // lanes per K/V row
    constexpr int RPW = 32 / LPR;  // rows per warp pass
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const long long wid = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int R = p.B * p.W;
    if (wid >= static_cast<long long>(R) * p.Hq) return;  // warp-uniform
    const int r = static_cast<int>(wid / p.Hq);
    const int h = static_cast<int>(wid % p.Hq);
    const int g = h / p.G;
    const int b = r / p.W;
    const int w = r % p.W;
    const int li = lane % LPR;
    const int rg = lane / LPR;

    const int* rq = p.req + b * kReqFields;
    const int P = __ldg(rq + kReqPrefix);
    const int T = __ldg(rq + kReqTail);
    const int nsplit = __ldg(rq + kReqSplits);
    const int part_off = __ldg(rq + kReqPartOff);
    const int ps_mask = (1 << p.ps_log2) - 1;

    const uint16_t* qbase = static_cast<const uint16_t*>(p.q) + (static_cast<long long>(r) * p.Hq + h) * D;
    float q[8];
    unpack8<BF16>(__ldg(reinterpret_cast<const uint4*>(qbase) + li), q);

    // ---- tail: online softmax per row group
    float m = -INFINITY, l = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const int passes = (T + RPW - 1) / RPW;
    for (int pass = 0; pass < passes; ++pass) {
        const int t = pass * RPW + rg;
        bool ok = t < T;
        long long row_off = 0;
        if (ok) {
            const int pos = P + t;
            const int src = __ldg(p.ci + (static_cast<long long>(b) * p.W + w) * p.max_seq + pos);
            ok = static_cast<unsigned>(src) < static_cast<unsigned>(p.W);
            int page = -1;
            if (ok) page = __ldg(p.beam_pages + (static_cast<long long>(b) * p.W + src) * p.beam_pages_stride +
                                 (pos >> p.ps_log2));
            ok = ok && static_cast<unsigned>(page) < static_cast<unsigned>(p.num_pages);
            if (!ok) {
                if (li == 0) atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
            } else {
                row_off = (((static_cast<long long>(page) * p.Hkv + g) << p.ps_log2) + (pos & ps_mask)) * D;
            }
        }
        float k[8], v[8];
        if (ok) {
            unpack8<BF16>(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_pool) + row_off) + li), k);
            unpack8<BF16>(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v_pool) + row_off) + li), v);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) k[e] = v[e] = 0.f;
        }
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) dot = fmaf(q[e], k[e], dot);
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) dot += __shfl_xor_sync(FULL, dot, off);
        if (ok) {
            const float s = dot * p.scale_log2;
            const float m_new = fmaxf(m, s);
            const float a = exp2f(m - m_new);  // m = -inf -> 0
            const float e_s = exp2f(s - m_new);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(acc[e], a, e_s * v[e]);
            l = fmaf(l, a, e_s);
            m = m_new;
        }
    }
    // combine the row groups of the warp
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
        const float mo = __shfl_xor_sync(FULL, m, off);
        const float lo = __shfl_xor_sync(FULL, l, off);
        float ao[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ao[e] = __shfl_xor_sync(FULL, acc[e], off);
        const float mn = fmaxf(m, mo);
        if (mn != -INFINITY) {
            const float fa = exp2f(m - mn), fo = exp2f(mo - mn);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = acc[e] * fa + ao[e] * fo;
            l = l * fa + lo * fo;
            m = mn;
        }
    }
    if (rg != 0) return;

    // ---- merge with the prompt partial states by log-sum-exp (base 2)
    const long long pstride = static_cast<long long>(p.W) * p.Hq;  // rows of one partial slot
    const long long prow = (static_cast<long long>(part_off) * p.W + w) * p.Hq + h;
    float Lmax = (l > 0.f) ? m + log2f(l) : -INFINITY;
    for (int s = 0; s < nsplit; ++s) Lmax = fmaxf(Lmax, __ldg(p.part_lse + prow + s * pstride));
    float out[8];
    float lse2;
    if (Lmax == -INFINITY) {
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = 0.f;
        lse2 = -INFINITY;
    } else {
        // tail weight exp2(m + log2 l - Lmax) times O_t = acc / l
        const float ft = (l > 0.f) ? exp2f(m - Lmax) : 0.f;
        float sum = l * ft;
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = acc[e] * ft;
        for (int s = 0; s < nsplit; ++s) {
            const float wgt = exp2f(__ldg(p.part_lse + prow + s * pstride) - Lmax);
            const float4* po = reinterpret_cast<const float4*>(p.part_o + (prow + s * pstride) * D) + li * 2;
            const float4 a0 = __ldg(po), a1 = __ldg(po + 1);
            out[0] = fmaf(wgt, a0.x, out[0]);
            out[1] = fmaf(wgt, a0.y, out[1]);
            out[2] = fmaf(wgt, a0.z, out[2]);
            out[3] = fmaf(wgt, a0.w, out[3]);
            out[4] = fmaf(wgt, a1.x, out[4]);
            out[5] = fmaf(wgt, a1.y, out[5]);
            out[6] = fmaf(wgt, a1.z, out[6]);
            out[7] = fmaf(wgt, a1.w, out[7]);
            sum += wgt;
        }
        const float inv = 1.f / sum;
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] *= inv;
        lse2 = Lmax + log2f(sum);
    }
    uint16_t* obase = static_cast<uint16_t*>(p.o) + (static_cast<long long>(r) * p.Hq + h) * D;
    reinterpret_cast<uint4*>(obase)[li] = pack8<BF16>(out);
    if (li == 0) p.lse[static_cast<long long>(r) * p.Hq + h] = p.lse_base2 ? lse2 : lse2 * 0.69314718055994530942f;
}

template <int D, bool BF16>
static cudaError_t launch_tail_t(const TailParams& p, cudaStream_t stream) {
    const long long warps = static_cast<long long>(p.B) * p.W * p.Hq;
    if (warps == 0) return cudaSuccess;
    const long long blocks = (warps + 3) / 4;
    tail_merge_kernel<D, BF16><<<static_cast<unsigned>(blocks), 128, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_tail(int head_dim, bool bf16, const TailParams& p, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return bf16 ? launch_tail_t<64, true>(p, stream) : launch_tail_t<64, false>(p, stream);
        case 128: return bf16 ? launch_tail_t<128, true>(p, stream) : launch_tail_t<128, false>(p, stream);
        case 256: return bf16 ? launch_tail_t<256, true>(p, stream) : launch_tail_t<256, false>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bsp
