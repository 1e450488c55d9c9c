// Paged KV append (TensorRT-LLM PR #18614, "Fuse MiniMax-M3 MSA per-layer
// KV-cache writes into one kernel", description): one launch writes the new
// token's K and V rows of every kv head at its flat slot, deriving
// (page, within-page offset) from out_cache_loc in registers.
//
// One thread moves one 16-byte chunk of K and the same chunk of V. Roofline:
// pure copy, algorithmic bytes = 2 (K, V) x 2 (read + write) x n x Hkv x D x 2.
#include <cuda_runtime.h>

#include "bsp_internal.h"
#include "../../include/bsp.h"

namespace bsp {

__global__ void __launch_bounds__(256) append_kv_kernel(AppendParams p) {
    const int chunks_per_head = p.D >> 3;
    const long long total = static_cast<long long>(p.n) * p.Hkv * chunks_per_head;
    const long long slots = static_cast<long long>(p.num_pages) << p.ps_log2;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(idx % chunks_per_head);
        const long long th = idx / chunks_per_head;
        const int h = static_cast<int>(th % p.Hkv);
        const long long i = th / p.Hkv;
        const int loc = __ldg(p.loc + i);
        if (loc < 0 || loc >= slots) {
            if (h == 0 && c == 0) atomicOr(p.status, BSP_DEVFLAG_PAGE_INDEX);
            continue;
        }
        const long long page = loc >> p.ps_log2;
        const long long off = loc & ((1 << p.ps_log2) - 1);
        const long long src = i * p.src_row_stride + static_cast<long long>(h) * p.D + c * 8;
        const long long dst = (((page * p.Hkv + h) << p.ps_log2) + off) * p.D + c * 8;
        const uint4 kv = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_new) + src));
        const uint4 vv = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v_new) + src));
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_pool) + dst) = kv;
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_pool) + dst) = vv;
    }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
    const long long total = static_cast<long long>(p.n) * p.Hkv * (p.D >> 3);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > 65535LL * 8) blocks = 65535LL * 8;
    append_kv_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace bsp
