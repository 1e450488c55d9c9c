// Rotary position embedding (RoPE) on the paged append. The pages rotate K by
// its position before the paged cache write (TensorRT-LLM PR #21738, review of
// flash_attn4_kernels.py: rope_write_kv_paged, with a partner lookup for partial
// rotary dims); RoPE itself is the published rotation (Su et al., RoFormer,
// section 3.2): pair j of the first rot dims turns by p * base^(-2j/rot).
//
// rope_append_kernel: the rows of one new token are its Hkv K rows (rotated,
// scattered into the pool), its Hkv V rows (copied into the pool) and, with q,
// its Hq query rows (rotated in place). A head row of D elements is D/8 16-byte
// chunks on D/8 consecutive lanes, so a warp moves 32 / (D/8) rows with one
// 16-byte load and one store per lane. In the rotate-half layout a chunk's
// partner (dims +- rot/2, rot a multiple of 16) sits on another lane of the
// same row and comes over by shuffle; in the interleaved layout both elements of
// a pair are in one chunk. cos/sin come from the fp32 table (L2-resident: all
// beams of a request share a position). Roofline: HBM copy, algorithmic bytes =
// n * (2 * Hkv * D * e (K, V read) + 2 * Hkv * D * e (pool rows written) +
// 2 * Hq * D * e (q read and written)) + 8 n (slots, positions) + the table rows
// of the distinct positions.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "bsp_internal.h"
#include "bsp_write.h"
#include "../../include/bsp.h"

namespace bsp {

namespace {

__device__ __forceinline__ float2 unpack2(uint32_t w, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
        return __bfloat1622float2(h);
    }
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
    uint32_t w;
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        w = *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        w = *reinterpret_cast<uint32_t*>(&h);
    }
    return w;
}

// 8 values times a multiplier, each product rounded to fp32, then to the nearest E4M3 (ties to even,
// saturating at +-448); byte e of the result holds value e
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float mul) {
    uint32_t w[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float2 a = make_float2(__fmul_rn(f[4 * e], mul), __fmul_rn(f[4 * e + 1], mul));
        const float2 b = make_float2(__fmul_rn(f[4 * e + 2], mul), __fmul_rn(f[4 * e + 3], mul));
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
        w[e] = (lo & 0xffffu) | (hi << 16);
    }
    return make_uint2(w[0], w[1]);
}

// x cos - y sin (sign = -1) or x cos + y sin (sign = +1): one product, one fused multiply-add
__device__ __forceinline__ float rot1(float x, float y, float c, float s, float sign) {
    return __fmaf_rn(x, c, sign * __fmul_rn(y, s));
}

}  // namespace

// FP8: K and V go to E4M3 pools: the rotated K values (fp32, before any 16-bit rounding) and the V
// values times their multipliers, quantised; q stays in its 16-bit dtype
template <int D, bool BF16, bool FP8>
__global__ void __launch_bounds__(256) rope_append_kernel(RopeAppendParams p) {
    constexpr int CPR = D / 8;     // 16-byte chunks per head row
    constexpr int RPW = 32 / CPR;  // head rows per warp
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int c = lane % CPR;
    const int seg = lane - c;  // first lane of this row's lane segment
    const long long warp = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int rpt = 2 * p.Hkv + (p.q ? p.Hq : 0);  // rows per token
    const long long gr = warp * RPW + lane / CPR;
    const bool live = gr < static_cast<long long>(p.n) * rpt;
    const long long i = live ? gr / rpt : 0;
    const int r = live ? static_cast<int>(gr % rpt) : 0;
    const bool is_k = r < p.Hkv;
    const bool is_v = !is_k && r < 2 * p.Hkv;
    const int h = is_k ? r : (is_v ? r - p.Hkv : r - 2 * p.Hkv);
    uint16_t* row;
    if (is_k || is_v)
        row = const_cast<uint16_t*>(static_cast<const uint16_t*>(is_k ? p.k_new : p.v_new)) + i * p.src_row_stride +
              static_cast<long long>(h) * D;
    else
        row = static_cast<uint16_t*>(p.q) + i * p.q_row_stride + static_cast<long long>(h) * D;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (live) x = (is_k || is_v) ? __ldcs(reinterpret_cast<const uint4*>(row) + c) : reinterpret_cast<const uint4*>(row)[c];
    int pos = 0, loc = 0;
    if (live) {
        pos = __ldg(p.pos + i);
        loc = __ldg(p.loc + i);
    }
    const long long slots = static_cast<long long>(p.num_pages) << p.ps_log2;
    const bool pos_ok = pos >= 0 && pos < p.max_pos;
    const bool loc_ok = loc >= 0 && loc < slots;
    const bool ok = live && pos_ok && loc_ok;
    const bool rotated = !is_v && 8 * c < p.rot;
    const int half = p.rot >> 1;
    uint4 y = x;
    float f[8];  // FP8: the chunk's values before quantisation
    if constexpr (FP8) {
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 a = unpack2(xw[u], BF16);
            f[2 * u] = a.x;
            f[2 * u + 1] = a.y;
        }
    }
    if (!p.interleaved) {
        // partner chunk of the rotate-half layout: c +- rot/16 (every lane takes part in the shuffles)
        const int hc = p.rot >> 4;
        const int src = seg + (8 * c < p.rot ? (c < hc ? c + hc : c - hc) : c);
        uint4 z;
        z.x = __shfl_sync(FULL, x.x, src);
        z.y = __shfl_sync(FULL, x.y, src);
        z.z = __shfl_sync(FULL, x.z, src);
        z.w = __shfl_sync(FULL, x.w, src);
        if (ok && rotated) {
            const bool first = c < hc;
            const int j0 = 8 * (first ? c : c - hc);
            const float* t = p.cos_sin + static_cast<long long>(pos) * p.rot;
            const float4 c0 = __ldg(reinterpret_cast<const float4*>(t + j0));
            const float4 c1 = __ldg(reinterpret_cast<const float4*>(t + j0 + 4));
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(t + half + j0));
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(t + half + j0 + 4));
            const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
            const float sign = first ? -1.f : 1.f;
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
            const uint32_t zw[4] = {z.x, z.y, z.z, z.w};
            uint32_t out[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 a = unpack2(xw[u], BF16);
                const float2 b = unpack2(zw[u], BF16);
                const float r0 = rot1(a.x, b.x, cs[2 * u], sn[2 * u], sign);
                const float r1 = rot1(a.y, b.y, cs[2 * u + 1], sn[2 * u + 1], sign);
                out[u] = pack2(r0, r1, BF16);
                if constexpr (FP8) {
                    f[2 * u] = r0;
                    f[2 * u + 1] = r1;
                }
            }
            y = make_uint4(out[0], out[1], out[2], out[3]);
        }
    } else if (ok && rotated) {
        // pairs (2j, 2j + 1) inside the chunk: frequencies 4c .. 4c + 3
        const float* t = p.cos_sin + static_cast<long long>(pos) * p.rot;
        const float4 c4 = __ldg(reinterpret_cast<const float4*>(t + 4 * c));
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(t + half + 4 * c));
        const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
        const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        uint32_t out[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 a = unpack2(xw[u], BF16);
            const float r0 = rot1(a.x, a.y, cs[u], sn[u], -1.f);
            const float r1 = rot1(a.y, a.x, cs[u], sn[u], 1.f);
            out[u] = pack2(r0, r1, BF16);
            if constexpr (FP8) {
                f[2 * u] = r0;
                f[2 * u + 1] = r1;
            }
        }
        y = make_uint4(out[0], out[1], out[2], out[3]);
    }
    if (!live) return;
    if (!ok) {
        if (r == 0 && c == 0) atomicOr(p.status, pos_ok ? BSP_DEVFLAG_PAGE_INDEX : BSP_DEVFLAG_POSITION);
        return;
    }
    if (is_k || is_v) {
        const long long page = loc >> p.ps_log2;
        const long long off = loc & ((1 << p.ps_log2) - 1);
        const long long dst = (((page * p.Hkv + h) << p.ps_log2) + off) * D;
        if constexpr (FP8) {
            uint8_t* pool = static_cast<uint8_t*>(is_k ? p.k_pool : p.v_pool);
            reinterpret_cast<uint2*>(pool + dst)[c] = quant8(f, is_k ? p.k_mul : p.v_mul);
        } else {
            uint16_t* pool = static_cast<uint16_t*>(is_k ? p.k_pool : p.v_pool);
            reinterpret_cast<uint4*>(pool + dst)[c] = y;
        }
    } else {
        reinterpret_cast<uint4*>(row)[c] = y;
    }
}

__global__ void rope_cos_sin_kernel(int max_pos, int rot, double base, float* cs) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int half = rot >> 1;
    if (t >= static_cast<long long>(max_pos) * half) return;
    const int pos = static_cast<int>(t / half);
    const int j = static_cast<int>(t % half);
    const double angle = static_cast<double>(pos) * pow(base, -2.0 * j / rot);
    double s, co;
    sincos(angle, &s, &co);
    cs[static_cast<long long>(pos) * rot + j] = __double2float_rn(co);
    cs[static_cast<long long>(pos) * rot + half + j] = __double2float_rn(s);
}

template <int D, bool BF16, bool FP8>
static cudaError_t launch_rope_t(const RopeAppendParams& p, cudaStream_t stream) {
    constexpr int RPW = 32 / (D / 8);
    const long long rows = static_cast<long long>(p.n) * (2 * p.Hkv + (p.q ? p.Hq : 0));
    if (rows == 0) return cudaSuccess;
    const long long warps = (rows + RPW - 1) / RPW;
    const long long blocks = (warps + 7) / 8;
    rope_append_kernel<D, BF16, FP8><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <bool FP8>
static cudaError_t launch_rope_d(int head_dim, bool bf16, const RopeAppendParams& p, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return bf16 ? launch_rope_t<64, true, FP8>(p, stream) : launch_rope_t<64, false, FP8>(p, stream);
        case 128: return bf16 ? launch_rope_t<128, true, FP8>(p, stream) : launch_rope_t<128, false, FP8>(p, stream);
        case 256: return bf16 ? launch_rope_t<256, true, FP8>(p, stream) : launch_rope_t<256, false, FP8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rope_append(int head_dim, bool bf16, bool fp8, const RopeAppendParams& p, cudaStream_t stream) {
    return fp8 ? launch_rope_d<true>(head_dim, bf16, p, stream) : launch_rope_d<false>(head_dim, bf16, p, stream);
}

template <bool FP8>
static const void* rope_fn(int head_dim, bool bf16) {
    switch (head_dim) {
        case 64: return bf16 ? (const void*)rope_append_kernel<64, true, FP8> : (const void*)rope_append_kernel<64, false, FP8>;
        case 128: return bf16 ? (const void*)rope_append_kernel<128, true, FP8> : (const void*)rope_append_kernel<128, false, FP8>;
        case 256: return bf16 ? (const void*)rope_append_kernel<256, true, FP8> : (const void*)rope_append_kernel<256, false, FP8>;
        default: return nullptr;
    }
}

// the same L1/shared split as the prompt kernel, so SMs are not reconfigured between the kernels of a step
cudaError_t prepare_rope_append(int head_dim, bool bf16, bool fp8) {
    const void* f = fp8 ? rope_fn<true>(head_dim, bf16) : rope_fn<false>(head_dim, bf16);
    if (!f) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_rope_cos_sin(int max_pos, int rot, double base, float* cos_sin, cudaStream_t stream) {
    const long long n = static_cast<long long>(max_pos) * (rot / 2);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    rope_cos_sin_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, stream>>>(max_pos, rot, base,
                                                                                                      cos_sin);
    return cudaGetLastError();
}

}  // namespace bsp
