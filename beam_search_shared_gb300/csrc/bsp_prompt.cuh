// Device-side pieces shared by the prompt-attention kernels (bsp_prefix.cu, bsp_wide.cu): the work
// unit as the plan image describes it, tile counts, and 16-bit packing.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "bsp_internal.h"

namespace bsp {

struct UnitInfo {
    int b, g, rb, part, P, page_off;
    int key_begin, key_end;  // keys [key_begin, key_end) of the request's prompt
    int T;                   // tail positions of the request
    bool fused;              // this kernel finishes the request: tail tiles when T > 0, final O / LSE
    int rows;                // the request's query rows per head (beams, or prompt tokens of a prefill)
    int causal;              // -1, or the cached rows C of a causal prefill: row t sees keys 0 .. C + t
    int row_off;             // the request's first row of q and o
};

__device__ __forceinline__ UnitInfo load_unit(const PrefixParams& p, int u) {
    const int4 a = __ldg(reinterpret_cast<const int4*>(p.units + static_cast<long long>(u) * kUnitFields));
    const int4 c = __ldg(reinterpret_cast<const int4*>(p.units + static_cast<long long>(u) * kUnitFields + 4));
    const int4 r = __ldg(reinterpret_cast<const int4*>(p.req + a.x * kReqFields));
    const int4 r2 = __ldg(reinterpret_cast<const int4*>(p.req + a.x * kReqFields + 4));
    const int4 r3 = __ldg(reinterpret_cast<const int4*>(p.req + a.x * kReqFields + 8));
    UnitInfo ui;
    ui.b = a.x;
    ui.g = a.y;
    ui.rb = a.z;
    ui.part = c.y;
    ui.P = r.x;
    ui.page_off = r2.x;
    ui.key_begin = a.w * kTileKeys;                // plan tiles are kTileKeys keys
    ui.key_end = min(c.x * kTileKeys, ui.P);
    ui.T = r.y;
    ui.fused = r2.y != 0;                            // kReqFused
    ui.rows = r3.x;                                  // kReqRows
    ui.causal = r3.y;                                // kReqCausal
    ui.row_off = r3.z;                               // kReqRowOff
    return ui;
}

// prompt tiles of a unit
template <int TK>
__device__ __forceinline__ int prompt_tiles(const UnitInfo& ui) {
    return (ui.key_end - ui.key_begin + TK - 1) / TK;
}

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

}  // namespace bsp
