// Device-side pieces shared by the prompt-attention kernels (bsp_prefix.cu, bsp_wide.cu, bsp_alt.cu): the
// work unit as the plan image describes it, tile counts, 16-bit packing, and the widening of E4M3 tiles.
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

// ---- E4M3 pools: the kernels load E4M3 tiles and widen them to the q dtype in shared memory

// Two E4M3 codes (bits 0-7 and 8-15 of `two`) as a pair of 16-bit floats of the q dtype, the first in the
// low half, exactly: every E4M3 value is a binary16 and a bfloat16 value. The hardware conversion gives
// binary16; for bfloat16 the binary16 sign, exponent and fraction fields move into bfloat16 fields (the
// exponent keeps its binary16 bias of 15 instead of 127: a factor 2^-112), and one multiplication by
// 2^112 restores the value. E4M3-derived binary16 values are zero or normal (the smallest, 2^-9, has
// exponent field 6), so the shifted bfloat16 value is zero or normal too and the product is exact.
template <bool BF16>
__device__ __forceinline__ uint32_t e4m3x2_to_16(uint32_t two) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
    if constexpr (!BF16) return h;
    // the fraction's low 7 bits are zero for these values, so nothing crosses from one half to the other
    const uint32_t t = ((h & 0x7fff7fffu) >> 3) | (h & 0x80008000u);
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x77807780u));  // 2^112 in both halves
    return r;
}
// 8 E4M3 codes (bytes in order) -> one 16-byte chunk of 8 16-bit values
template <bool BF16>
__device__ __forceinline__ uint4 e4m3x8_to_16(uint2 in) {
    return make_uint4(e4m3x2_to_16<BF16>(in.x & 0xffffu), e4m3x2_to_16<BF16>(in.x >> 16),
                      e4m3x2_to_16<BF16>(in.y & 0xffffu), e4m3x2_to_16<BF16>(in.y >> 16));
}

// Byte offset of 16-byte chunk kc (8 elements) of key row r in a 16-bit K or V tile of TK rows laid out
// as a TMA box with 128-byte swizzle: column half kc / 8, then row r, then chunk (kc % 8) ^ (r % 8).
template <int TK>
__device__ __forceinline__ uint32_t sw128_chunk(int kc, int r) {
    return static_cast<uint32_t>((kc >> 3) * (TK * 128) + r * 128 + (((kc & 7) ^ (r & 7)) << 4));
}

// Widens the E4M3 K or V tile that a TMA load left in the upper half of a ring slot (TK rows of D codes,
// row r at slot + TK * D + r * D) into the slot's 16-bit layout (sw128_chunk); rows >= valid become zero
// rows. Run by the NT threads gtid = 0 .. NT - 1 (NT = 64 or 128) of NT / 32 warps, which synchronise on
// named barrier `bar` (NT threads) at head_dim 64. The 16-bit rows overwrite the E4M3 rows in place:
//  - D = 128: a 16-bit row's first column half lies below the E4M3 rows and its second half on the E4M3
//    row of the same key, so each key row belongs to one warp (rows r with r mod (NT / 8) in the warp's
//    four values), which reads all of it before writing it;
//  - D = 64: the 16-bit row r covers E4M3 rows 2r - TK and 2r - TK + 1, so all threads read the whole
//    tile into registers before any of them writes.
// The caller fences the writes for the tensor core and synchronises the NT threads afterwards.
template <int D, int TK, bool BF16, int NT = 64>
__device__ __forceinline__ void widen_e4m3_tile(uint8_t* slot, int valid, int gtid, int bar) {
    static_assert(D == 64 || D == 128, "E4M3 tiles at head_dim 64 and 128");
    static_assert(NT == 64 || NT == 128, "64 or 128 threads");
    const uint8_t* src = slot + TK * D;
    if constexpr (D == 128) {
        constexpr int RS = NT / 8;  // rows one pass of the threads covers
        const int j = gtid & 7;     // codes 16j .. 16j + 15 of a row
        const int r0 = gtid >> 3;   // rows r0 + RS i: warp w holds r0 in [4w, 4w + 4)
#pragma unroll 1
        for (int i0 = 0; i0 < TK / RS; i0 += 4) {
            uint4 in[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = r0 + RS * (i0 + u);
                in[u] = r < valid ? *reinterpret_cast<const uint4*>(src + r * D + 16 * j) : make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = r0 + RS * (i0 + u);
                uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                if (r < valid) {
                    lo = e4m3x8_to_16<BF16>(make_uint2(in[u].x, in[u].y));
                    hi = e4m3x8_to_16<BF16>(make_uint2(in[u].z, in[u].w));
                }
                *reinterpret_cast<uint4*>(slot + sw128_chunk<TK>(2 * j, r)) = lo;
                *reinterpret_cast<uint4*>(slot + sw128_chunk<TK>(2 * j + 1, r)) = hi;
            }
            __syncwarp();
        }
    } else {
        constexpr int RS = NT / 4;  // rows one pass of the threads covers
        const int j = gtid & 3;     // codes 16j .. 16j + 15 of a row
        const int r0 = gtid >> 2;   // rows r0 + RS i
        uint4 in[TK / RS];
#pragma unroll
        for (int i = 0; i < TK / RS; ++i) {
            const int r = r0 + RS * i;
            in[i] = r < valid ? *reinterpret_cast<const uint4*>(src + r * D + 16 * j) : make_uint4(0, 0, 0, 0);
        }
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(NT) : "memory");
#pragma unroll
        for (int i = 0; i < TK / RS; ++i) {
            const int r = r0 + RS * i;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (r < valid) {
                lo = e4m3x8_to_16<BF16>(make_uint2(in[i].x, in[i].y));
                hi = e4m3x8_to_16<BF16>(make_uint2(in[i].z, in[i].w));
            }
            *reinterpret_cast<uint4*>(slot + sw128_chunk<TK>(2 * j, r)) = lo;
            *reinterpret_cast<uint4*>(slot + sw128_chunk<TK>(2 * j + 1, r)) = hi;
        }
    }
}

}  // namespace bsp
