// Paged KV append (TensorRT-LLM PR #18614, "Fuse MiniMax-M3 MSA per-layer
// KV-cache writes into one kernel", description): one launch writes the new
// token's K and V rows of every kv head at its flat slot, deriving
// (page, within-page offset) from out_cache_loc in registers.
//
// One warp per (new token, kv head): the slot is read once per warp, and the
// warp's lanes move the head's K row and V row (D/8 16-byte chunks each) with
// one load and one store per chunk, so every lane has its loads in flight at
// once. Roofline: pure copy, algorithmic bytes = 2 (K, V) x 2 (read + write) x
// n x Hkv x D x 2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "bsp_internal.h"
#include "bsp_write.h"
#include "../../include/bsp.h"

namespace bsp {

__global__ void __launch_bounds__(256) append_kv_kernel(AppendParams p) {
    const int lane = threadIdx.x & 31;
    const long long wi = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wi >= static_cast<long long>(p.n) * p.Hkv) return;
    const long long i = wi / p.Hkv;
    const int h = static_cast<int>(wi % p.Hkv);
    const int cpr = p.D >> 3;  // 16-byte chunks per row
    const uint16_t* ks = static_cast<const uint16_t*>(p.k_new) + i * p.src_row_stride + static_cast<long long>(h) * p.D;
    const uint16_t* vs = static_cast<const uint16_t*>(p.v_new) + i * p.src_row_stride + static_cast<long long>(h) * p.D;
    // loads first (they do not depend on the slot), then the slot check and the stores
    uint4 val[2];
    int idx[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        idx[u] = u * 32 + lane;  // chunk index over [K row | V row]
        if (idx[u] < 2 * cpr) {
            const bool is_v = idx[u] >= cpr;
            const int c = is_v ? idx[u] - cpr : idx[u];
            val[u] = __ldcs(reinterpret_cast<const uint4*>(is_v ? vs : ks) + c);
        }
    }
    const int loc = __ldg(p.loc + i);
    const long long slots = static_cast<long long>(p.num_pages) << p.ps_log2;
    if (loc < 0 || loc >= slots) {
        if (lane == 0 && h == 0) atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
        return;
    }
    const long long page = loc >> p.ps_log2;
    const long long off = loc & ((1 << p.ps_log2) - 1);
    const long long dst = (((page * p.Hkv + h) << p.ps_log2) + off) * p.D;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        if (idx[u] < 2 * cpr) {
            const bool is_v = idx[u] >= cpr;
            const int c = is_v ? idx[u] - cpr : idx[u];
            uint16_t* pool = static_cast<uint16_t*>(is_v ? p.v_pool : p.k_pool);
            reinterpret_cast<uint4*>(pool + dst)[c] = val[u];
        }
    }
}

// the same L1/shared split as the prompt kernel, so SMs are not reconfigured between the
// kernels of a step
cudaError_t prepare_append() {
    return cudaFuncSetAttribute(append_kv_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
    const long long warps = static_cast<long long>(p.n) * p.Hkv;
    if (warps == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (warps + (threads / 32) - 1) / (threads / 32);
    append_kv_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    return cudaGetLastError();
}

// Append into E4M3 pools (the KV write of a cache kept in fp8: TensorRT-LLM PR #18614, the review
// follow-up commit on the fused KV write: an fp8 source written into an fp8 cache, and the
// source/cache dtype conversion of the fused write). The same warp per (new token, kv head) as the
// plain append. A 16-bit source element becomes the E4M3 value nearest to its fp32 product with the
// tensor's multiplier (ties to even, saturating at +-448): a lane converts one 16-byte chunk of 8
// elements into 8 bytes. An E4M3 source row is copied in 16-byte chunks. Roofline: algorithmic bytes =
// 2 (K, V) x n x Hkv x D x (source element size + 1).
template <int SRC>
__global__ void __launch_bounds__(256) append_kv_fp8_kernel(AppendFp8Params p) {
    const int lane = threadIdx.x & 31;
    const long long wi = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wi >= static_cast<long long>(p.n) * p.Hkv) return;
    const long long i = wi / p.Hkv;
    const int h = static_cast<int>(wi % p.Hkv);
    constexpr int ES = SRC == 2 ? 1 : 2;           // source element bytes
    const int cpr = p.D * ES / 16;                 // 16-byte source chunks per row
    const uint8_t* ks = static_cast<const uint8_t*>(p.k_new) + (i * p.src_row_stride + static_cast<long long>(h) * p.D) * ES;
    const uint8_t* vs = static_cast<const uint8_t*>(p.v_new) + (i * p.src_row_stride + static_cast<long long>(h) * p.D) * ES;
    uint4 val[4];
    int idx[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        idx[u] = u * 32 + lane;  // chunk index over [K row | V row]
        if (idx[u] < 2 * cpr) {
            const bool is_v = idx[u] >= cpr;
            const int c = is_v ? idx[u] - cpr : idx[u];
            val[u] = __ldcs(reinterpret_cast<const uint4*>(is_v ? vs : ks) + c);
        }
    }
    const int loc = __ldg(p.loc + i);
    const long long slots = static_cast<long long>(p.num_pages) << p.ps_log2;
    if (loc < 0 || loc >= slots) {
        if (lane == 0 && h == 0) atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
        return;
    }
    const long long page = loc >> p.ps_log2;
    const long long off = loc & ((1 << p.ps_log2) - 1);
    const long long dst = (((page * p.Hkv + h) << p.ps_log2) + off) * p.D;  // bytes
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (idx[u] < 2 * cpr) {
            const bool is_v = idx[u] >= cpr;
            const int c = is_v ? idx[u] - cpr : idx[u];
            uint8_t* pool = (is_v ? p.v_pool : p.k_pool) + dst;
            if constexpr (SRC == 2) {
                reinterpret_cast<uint4*>(pool)[c] = val[u];
            } else {
                const float mul = is_v ? p.v_mul : p.k_mul;
                const uint32_t w[4] = {val[u].x, val[u].y, val[u].z, val[u].w};
                uint32_t q[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float2 a, b;
                    if constexpr (SRC == 0) {
                        a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * e]));
                        b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * e + 1]));
                    } else {
                        a = __half22float2(*reinterpret_cast<const __half2*>(&w[2 * e]));
                        b = __half22float2(*reinterpret_cast<const __half2*>(&w[2 * e + 1]));
                    }
                    a = make_float2(__fmul_rn(a.x, mul), __fmul_rn(a.y, mul));
                    b = make_float2(__fmul_rn(b.x, mul), __fmul_rn(b.y, mul));
                    const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
                    const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
                    q[e] = (lo & 0xffffu) | (hi << 16);
                }
                reinterpret_cast<uint2*>(pool)[c] = make_uint2(q[0], q[1]);
            }
        }
    }
}

cudaError_t prepare_append_fp8(int src) {
    const void* f = src == 0 ? (const void*)append_kv_fp8_kernel<0>
                  : src == 1 ? (const void*)append_kv_fp8_kernel<1>
                             : (const void*)append_kv_fp8_kernel<2>;
    return cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_append_fp8(int src, const AppendFp8Params& p, cudaStream_t stream) {
    const long long warps = static_cast<long long>(p.n) * p.Hkv;
    if (warps == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = static_cast<unsigned>((warps + (threads / 32) - 1) / (threads / 32));
    switch (src) {
        case 0: append_kv_fp8_kernel<0><<<blocks, threads, 0, stream>>>(p); break;
        case 1: append_kv_fp8_kernel<1><<<blocks, threads, 0, stream>>>(p); break;
        case 2: append_kv_fp8_kernel<2><<<blocks, threads, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace bsp
