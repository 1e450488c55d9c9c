// Internal contract between the host library (bsp_host.cpp) and the kernels:
// the staged plan image layout and the launch parameter blocks.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/bsp.h"

namespace bsp {

// Prompt-attention tiling.
constexpr int kTileKeys = 64;      // keys per prompt tile (MMA N of Q*K^T, MMA K of P*V)
constexpr int kRowsPerBlock = 128; // query rows per CTA (MMA M)
constexpr int kExtraParts = 64;    // key splits beyond one per request the workspace holds

// Device workspace: [status words | plan image | partial LSE | partial O].
constexpr size_t kStatusBytes = 256;
constexpr size_t kAlign = 256;

// Plan image (int32 fields, offsets relative to the image start).
constexpr int kImageHeaderBytes = 64;  // u64 generation, i32 batch, i32 num_units, ...
// Per-request record.
// kReqFused: the prompt kernel finishes the request (one prompt partial state, and every unit's tail keys
// fit the prompt kernel's tail tiles); the tail kernel skips it.
// kReqRows: the request's query rows per (kv head, head in group) - beams for a decode step, prompt
// tokens for a prefill; kReqRowOff: its first row of q / o (b * W, or the tokens of earlier requests);
// kReqCausal: -1, or the cached rows C of a causal prefill (row t sees keys 0 .. C + t).
enum ReqField { kReqPrefix = 0, kReqTail = 1, kReqSplits = 2, kReqPartOff = 3, kReqPageOff = 4, kReqFused = 5,
                kReqRows = 8, kReqCausal = 9, kReqRowOff = 10, kReqFields = 12 };
// keys per tile of the prompt kernel, which bounds a row block's tail keys for the fused tail
constexpr int prefix_tile_keys(int head_dim) { return head_dim <= 128 ? 128 : 64; }
// tail tiles of prefix_tile_keys(head_dim) keys the one-set prompt kernel may gather for a unit (the
// request is finished by the tail kernel beyond)
constexpr int kPrefixMaxTailTiles = 4;
// Beams per TMEM lane quadrant when the prompt kernel places a row block's query rows in lanes
// 0-15 of each quadrant and gives each row two softmax threads (half of the keys each): the
// block's beams spread over the four quadrants, at most 16 rows each, with 128-key tiles. 0 when
// the block does not fit that way (the rows then fill the lanes densely, one thread per row).
constexpr int prefix_quad_beams(int head_dim, int beams_per_block, int group) {
    const int bq = (beams_per_block + 3) / 4;
    return (prefix_tile_keys(head_dim) == 128 && bq * group <= 16) ? bq : 0;
}
// The wide layout of a decode step (bsp_wide.cu): when a (request, kv head) has more query rows than
// one MMA holds (W * G in (128, 256]) at head_dim <= 128, one unit holds all of them as two M = 128
// blocks (beams [0, Wb) and [Wb, W), Wb = ceil(W / 2)) that share every K/V tile, so the prompt is read
// once. Each block's beams spread over the four TMEM lane quadrants, bq = ceil(Wb / 4) beams (bq * G
// rows) per quadrant. 0 when the beams do not fit that way.
constexpr int wide_quad_beams(int head_dim, int beam_width, int group) {
    const int wb = (beam_width + 1) / 2;
    const int bq = (wb + 3) / 4;
    return (head_dim <= 128 && beam_width * group > kRowsPerBlock && beam_width * group <= 2 * kRowsPerBlock &&
            bq * group <= 32)
               ? bq
               : 0;
}
// tail tiles of 128 keys a wide unit may gather (the request is finished by the tail kernel beyond)
constexpr int kWideMaxTailTiles = 4;
// The alternating-tile layout of a decode step (bsp_alt.cu), at head_dim <= 128: a unit is one query-row
// block (W_blk beams x G heads <= 128 rows) whose key tiles go alternately to two softmax warp sets;
// the block's beams spread over the four TMEM lane quadrants, bq = ceil(W_blk / 4) beams (bq * G rows)
// per quadrant. 0 when the beams do not fit that way.
constexpr int alt_quad_beams(int head_dim, int beams_per_block, int group) {
    const int bq = (beams_per_block + 3) / 4;
    return (head_dim <= 128 && beams_per_block * group <= kRowsPerBlock && bq * group <= 32) ? bq : 0;
}
// tail tiles of 128 keys an alternating-tile unit may gather (the request is finished by the tail
// kernel beyond)
constexpr int kAltMaxTailTiles = 4;
// Per-work-unit record: request, kv head, query-row block, key tiles [kt0, kt1), partial slot, and
// the cost the host dealt it by (eighths of a prompt-kernel key tile; not read by the kernels).
enum UnitField { kUnitReq = 0, kUnitKvHead = 1, kUnitRowBlock = 2, kUnitTile0 = 3, kUnitTile1 = 4, kUnitPart = 5,
                 kUnitCost = 6, kUnitFields = 8 };

struct PrefixParams {
    // fused requests: tail keys gathered by the prompt kernel, final O / LSE written by it
    const void* k_pool;
    const void* v_pool;
    const int32_t* beam_pages;
    const int32_t* ci;
    void* o;
    float* lse;
    int beam_pages_stride, max_seq, lse_base2;
    const int32_t* units;    // [num_units][kUnitFields], grouped by CTA
    const int32_t* cta_off;  // [gridDim.x + 1]: CTA c runs units cta_off[c] .. cta_off[c+1]-1
    const int32_t* req;
    const int32_t* pages;
    float* part_o;    // [part][W][Hq][D]   (normalised partial output)
    float* part_lse;  // [part][W][Hq]      (log2-sum-exp2 of the scaled scores)
    int32_t* status;
    int W, Hq, Hkv, G, ps_log2, Wblk, num_pages;
    int bq;            // > 0: half-row softmax, bq beams of the block per TMEM lane quadrant (prefix_quad_beams)
    int num_units;     // units in the list
    float v_scale;     // E4M3 pools: the values' per-tensor scale, applied to O (1 for 16-bit pools)
    // graph mode (else null): the staged plan's header, checked at the start against the launch
    // (batch, beam width, one CTA per SM of the plan, a decode plan)
    const int32_t* graph_hdr;
    int graph_batch;
    float scale_log2;  // softmax_scale * log2(e)
};

struct TailParams {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* beam_pages;
    const int32_t* ci;
    const int32_t* req;
    const float* part_o;
    const float* part_lse;
    void* o;
    float* lse;
    int32_t* status;
    int B, W, Hq, Hkv, G, ps_log2, num_pages, beam_pages_stride, max_seq;
    float scale_log2;
    int lse_base2;
    float v_scale;     // E4M3 pools: the values' per-tensor scale, applied to the tail's O (1 otherwise)
    // graph mode (else null): the staged plan's header, checked against the launch (batch, beam width,
    // a decode plan, a tail bound within the one the launch was made for)
    const int32_t* graph_hdr;
    int graph_max_tail;
};

struct AppendParams {
    const void* k_new;
    const void* v_new;
    int64_t src_row_stride;  // elements
    const int32_t* loc;
    void* k_pool;
    void* v_pool;
    int32_t* status;
    int n, Hkv, D, ps_log2, num_pages;
};

cudaError_t launch_prefix(int head_dim, bool bf16, int ctas, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const PrefixParams& p, cudaStream_t stream);
// Kernel attributes (shared-memory size and split) are set by the prepare_* calls, once before
// the launches, so that timing events recorded around a launch bracket the launch alone.
cudaError_t prepare_prefix(int head_dim, bool bf16);
cudaError_t prepare_tail(int head_dim, bool bf16, int max_tail_len, int num_q_heads, bool fp8 = false);
// after_prefix: the prompt kernel was the last launch on `stream`; the tail kernel is then a
// programmatic dependent launch of it (it starts on SMs the prompt kernel has left, resolves and
// prefetches its tail rows, and waits for the prompt kernel's partials before merging).
cudaError_t launch_tail(int head_dim, bool bf16, int max_tail_len, const TailParams& p, bool after_prefix,
                        cudaStream_t stream, bool fp8 = false);
// The alternating-tile prompt kernel (p.Wblk = beams per row block, p.bq = beams per quadrant). fp8: E4M3
// pools (tk, tv map one-byte elements without swizzle, boxes of min(page, 64) rows x head_dim bytes).
cudaError_t prepare_alt(int head_dim, bool bf16, bool fp8 = false);
cudaError_t launch_alt(int head_dim, bool bf16, int ctas, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const PrefixParams& p, cudaStream_t stream, bool fp8 = false);
// The wide-layout prompt kernel (p.Wblk = beams per block, p.bq = beams per quadrant); fp8 as above.
cudaError_t prepare_wide(int head_dim, bool bf16, bool fp8 = false);
cudaError_t launch_wide(int head_dim, bool bf16, int ctas, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const PrefixParams& p, cudaStream_t stream, bool fp8 = false);
cudaError_t prepare_append();
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// bsp_host.cpp: the attention of a plan whose status word, image and partial states sit at `ws`
// (the caller's workspace, or the fixed scratch of the no-allocation entry point). attn_check_args
// checks what the host can check and enqueues nothing; attn_launches enqueues the launches.
// fp8: the caller is the E4M3 entry point (the plan's pools must then be E4M3, and 16-bit otherwise);
// k_scale and v_scale are the E4M3 pools' per-tensor scales (1 for 16-bit pools).
bsp_status attn_check_args(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
                           int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse, bool prefill,
                           bool fp8 = false, float k_scale = 1.f, float v_scale = 1.f);
bsp_status attn_launches(const bsp_plan_t* plan, uint8_t* ws, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
                         int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse,
                         void* const* events, cudaStream_t s, bool prefill, float k_scale = 1.f, float v_scale = 1.f);
// A decode plan with the packed layout (sections and partial states sized by the plan's own units and
// splits), for a caller that never replays it from a CUDA graph.
bsp_status plan_build_packed(const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len,
                             const int32_t* tail_len, const int32_t* prefix_pages, int32_t prefix_pages_stride,
                             int32_t max_tail, int32_t num_sms, void* image, size_t image_bytes, bsp_plan_t* out);

}  // namespace bsp
