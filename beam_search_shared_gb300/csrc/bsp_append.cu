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
#include <cuda_runtime.h>

#include "bsp_internal.h"
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

}  // namespace bsp
