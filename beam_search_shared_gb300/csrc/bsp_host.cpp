// Host side of libbsp.so: argument validation, per-step planning, plan
// staging without a stream sync, tensor-map encoding and kernel launches.
// Everything here is declared in include/bsp.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <limits>
#include <queue>
#include <utility>
#include <thread>
#include <vector>

#include "../../include/bsp.h"
#include "bsp_internal.h"
#include "bsp_write.h"

namespace {

using namespace bsp;

constexpr uint64_t kStagingMagic = 0x3150534250534253ull;
constexpr size_t kStagingHeaderBytes = 256;

// First bytes of the caller's host staging buffer.
struct StagingHeader {
    uint64_t magic;
    uint64_t generation;     // latest plan staged through this buffer
    uint64_t echoed[2];      // generation whose image copy from slot i has executed (written by the stream)
    uint64_t ws_device;      // device workspace this buffer is paired with
    uint64_t slot_bytes;     // bytes of each of the two image slots that follow the header
};
static_assert(sizeof(StagingHeader) <= kStagingHeaderBytes, "staging header");

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bsp_status check_geometry(const bsp_geometry* geo) {
    if (!geo) return BSP_ERR_INVALID_ARG;
    if (geo->dtype != BSP_DTYPE_BF16 && geo->dtype != BSP_DTYPE_FP16) return BSP_ERR_UNSUPPORTED;
    if (geo->kv_dtype != BSP_KV_DTYPE_SAME && geo->kv_dtype != BSP_KV_DTYPE_E4M3) return BSP_ERR_UNSUPPORTED;
    if (geo->head_dim != 64 && geo->head_dim != 128 && geo->head_dim != 256) return BSP_ERR_UNSUPPORTED;
    if (geo->num_q_heads <= 0 || geo->num_kv_heads <= 0 || geo->num_pages <= 0) return BSP_ERR_INVALID_ARG;
    if (geo->num_q_heads % geo->num_kv_heads != 0) return BSP_ERR_UNSUPPORTED;
    if (geo->num_q_heads / geo->num_kv_heads > BSP_MAX_GROUP) return BSP_ERR_UNSUPPORTED;
    if (!is_pow2(geo->page_size) || geo->page_size < 8 || geo->page_size > 128) return BSP_ERR_UNSUPPORTED;
    // pool rows are addressed with 32-bit TMA coordinates
    if (static_cast<int64_t>(geo->num_pages) * geo->num_kv_heads * geo->page_size >= (int64_t(1) << 31))
        return BSP_ERR_UNSUPPORTED;
    return BSP_OK;
}

// Query rows of one (request, kv head) are W*G; a CTA takes whole beams, at most 128 rows.
void row_blocks(int W, int G, int* nrb, int* wblk) {
    const int wmax = std::max(1, kRowsPerBlock / G);
    const int n = static_cast<int>(ceil_div(W, wmax));
    *nrb = n;
    *wblk = static_cast<int>(ceil_div(W, n));
}

struct DeviceLayout {
    size_t image, part_lse, part_o, total;
};

// CTA-table entries the workspace reserves beyond the units (a plan's table has num_sms + 1 entries)
constexpr int64_t kMaxCtas = 1024;

DeviceLayout device_layout(size_t image_bytes, int64_t parts, int W, const bsp_geometry& geo) {
    DeviceLayout L;
    L.image = align_up(image_bytes, kAlign);
    L.part_lse = align_up(static_cast<size_t>(parts) * W * geo.num_q_heads * sizeof(float), kAlign);
    L.part_o = align_up(static_cast<size_t>(parts) * W * geo.num_q_heads * geo.head_dim * sizeof(float), kAlign);
    L.total = kStatusBytes + L.image + L.part_lse + L.part_o;
    return L;
}

bool plan_is_current(const bsp_plan_t* plan) {
    if (!plan->ws_host || !plan->ws_device || plan->generation == 0) return false;
    const StagingHeader* hdr = static_cast<const StagingHeader*>(plan->ws_host);
    return hdr->magic == kStagingMagic && hdr->generation == plan->generation &&
           hdr->ws_device == reinterpret_cast<uint64_t>(plan->ws_device);
}

bsp_status check_plan(const bsp_plan_t* plan) {
    if (!plan) return BSP_ERR_INVALID_ARG;
    if (plan->generation == 0 || !plan->ws_device || !plan->ws_host) return BSP_ERR_INVALID_ARG;
    if (!plan_is_current(plan)) return BSP_ERR_STALE_PLAN;
    return check_geometry(&plan->geo);
}

// Device memory (or managed) pointer, 16-byte aligned.
bool device_ptr_ok(const void* p) {
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A tiled tensor map of 16-bit elements with 128-byte swizzle (the MMA operand layout), or with
// e4m3 = true of one-byte elements without swizzle (E4M3 tiles that the kernel widens itself).
bool encode_map(CUtensorMap* m, int dtype, int rank, const void* base, const cuuint64_t* dims,
                const cuuint64_t* strides_bytes, const cuuint32_t* box, bool e4m3 = false) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapDataType t = e4m3                     ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : dtype == BSP_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(m, t, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides_bytes, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, e4m3 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Records a timing event; under stream capture it becomes an external event-record node.
bool record_event(void* const* events, int i, cudaStream_t s) {
    if (!events) return true;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return false;
    cudaEvent_t ev = static_cast<cudaEvent_t>(events[i]);
    if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal) == cudaSuccess;
    return cudaEventRecord(ev, s) == cudaSuccess;
}

}  // namespace

extern "C" {

const char* bsp_status_string(int32_t status) {
    switch (status) {
        case BSP_OK: return "ok";
        case BSP_ERR_INVALID_ARG: return "invalid argument";
        case BSP_ERR_UNSUPPORTED: return "unsupported configuration";
        case BSP_ERR_PAGE_INDEX: return "page index, slot or indirection value out of range";
        case BSP_ERR_CAPACITY: return "workspace, staging buffer or tail bound too small";
        case BSP_ERR_STALE_PLAN: return "stale plan (superseded by a newer plan on this workspace)";
        case BSP_ERR_CUDA: return "CUDA call failed";
        case BSP_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait expired";
        default: return "unknown status";
    }
}

int32_t bsp_bucket_rows(int32_t valid_rows, int32_t capacity) {
    if (capacity < 1) return -1;
    if (valid_rows <= 0) return 1;
    const int64_t r = ceil_div(valid_rows, 256) * 256;
    return r < capacity ? static_cast<int32_t>(r) : capacity;
}

bsp_status bsp_workspace_size(const bsp_geometry* geo, int32_t max_batch, int32_t max_beam, int32_t max_prefix_pages,
                              size_t* device_bytes, size_t* host_bytes) {
    bsp_status st = check_geometry(geo);
    if (st != BSP_OK) return st;
    if (max_batch < 0 || max_beam < 1 || max_prefix_pages < 0 || !device_bytes || !host_bytes)
        return BSP_ERR_INVALID_ARG;
    const int G = geo->num_q_heads / geo->num_kv_heads;
    int nrb, wblk;
    row_blocks(max_beam, G, &nrb, &wblk);
    // E4M3 pools: row blocks of at most 4 * floor(32 / G) beams (the planner's bound for those kernels)
    if (geo->kv_dtype == BSP_KV_DTYPE_E4M3) nrb = std::max(nrb, static_cast<int>(ceil_div(max_beam, 4 * (32 / G))));
    const int64_t parts_cap = static_cast<int64_t>(max_batch) + kExtraParts;
    const int64_t units_max = parts_cap * geo->num_kv_heads * nrb;
    const size_t image = kImageHeaderBytes + static_cast<size_t>(max_batch) * kReqFields * 4 +
                         static_cast<size_t>(units_max) * kUnitFields * 4 +
                         (static_cast<size_t>(std::max<int64_t>(units_max, kMaxCtas)) + 1) * 4 +
                         static_cast<size_t>(max_batch) * max_prefix_pages * 4;
    DeviceLayout L = device_layout(image, parts_cap, max_beam, *geo);
    *device_bytes = L.total;
    *host_bytes = kStagingHeaderBytes + 2 * L.image;
    return BSP_OK;
}

}  // extern "C"

namespace {
// A prefill plan: request b holds cached_len[b] valid cached rows and prompt_len[b] prompt tokens.
struct PrefillSpec {
    const int32_t* cached_len;
    const int32_t* prompt_len;
    bool causal;
    bool splits;  // key splits of the cached rows allowed (partial states the tail kernel merges)
};

// Whether the prompt kernel of plan layout `layout` finishes a decode request: its prompt is one partial
// state (nsplit == 1) and the tail keys of one unit's beams (wblk of them; all W for the wide kernel) fit
// the kernel's tail tiles: up to 4 tiles of 128 keys (layouts 1 and 2), up to 4 prompt tiles (layout 0:
// 128 keys, 64 at head_dim 256).
int64_t request_tail_tiles(int layout, int head_dim, int wblk, int32_t tail) {
    return ceil_div(static_cast<int64_t>(tail) * wblk, layout ? 128 : prefix_tile_keys(head_dim));
}
bool request_fused(int layout, int head_dim, int wblk, int32_t nsplit, int32_t tail) {
    return nsplit == 1 && request_tail_tiles(layout, head_dim, wblk, tail) <=
                              (layout == 1 ? kAltMaxTailTiles : layout == 2 ? kWideMaxTailTiles : kPrefixMaxTailTiles);
}

// The plan image of a decode step (pf == nullptr: prefix_len / tail_len per request, beam_width rows
// each) or of a prefill (pf: the prompt tokens are the rows, the keys are the cached rows and the
// prompt, no tail; a request whose units are much longer than the mean CTA load has its cached rows
// split into key ranges whose partial states the tail kernel merges, the others are finished by the
// prompt kernel).
bsp_status plan_build_core(const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len_in,
                           const int32_t* tail_len_in, const int32_t* prefix_pages, int32_t prefix_pages_stride,
                           int32_t max_tail, int32_t num_sms, void* image, size_t image_bytes, bsp_plan_t* out,
                           const PrefillSpec* pf, bool fixed_layout = true) {
    bsp_status st = check_geometry(geo);
    if (st != BSP_OK) return st;
    if (!out || batch < 0 || beam_width < 1 || num_sms < 1 || prefix_pages_stride < 0) return BSP_ERR_INVALID_ARG;
    if (num_sms > kMaxCtas) return BSP_ERR_UNSUPPORTED;
    if (max_tail < 0) return BSP_ERR_INVALID_ARG;
    if (max_tail > BSP_MAX_TAIL) return BSP_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(batch) * beam_width > (int64_t(1) << 30)) return BSP_ERR_UNSUPPORTED;
    if (batch > 0 && !pf && (!prefix_len_in || !tail_len_in)) return BSP_ERR_INVALID_ARG;
    if (batch > 0 && pf && (!pf->cached_len || !pf->prompt_len)) return BSP_ERR_INVALID_ARG;
    const int ps = geo->page_size;
    const int G = geo->num_q_heads / geo->num_kv_heads;
    const int Hkv = geo->num_kv_heads;
    // per request: keys, tail, query rows, causal base, first row
    std::vector<int32_t> pl(batch), tl(batch), rows(batch), causal(batch), row_off(batch);
    int64_t total_rows = 0;
    for (int b = 0; b < batch; ++b) {
        if (pf) {
            const int64_t c = pf->cached_len[b], sq = pf->prompt_len[b];
            if (c < 0 || sq < 0) return BSP_ERR_INVALID_ARG;
            if (c + sq > (1 << 30)) return BSP_ERR_UNSUPPORTED;
            pl[b] = sq > 0 ? static_cast<int32_t>(c + sq) : 0;  // no rows: nothing to attend
            tl[b] = 0;
            rows[b] = static_cast<int32_t>(sq);
            causal[b] = pf->causal ? static_cast<int32_t>(c) : -1;
        } else {
            pl[b] = prefix_len_in[b];
            tl[b] = tail_len_in[b];
            rows[b] = beam_width;
            causal[b] = -1;
        }
        if (total_rows + rows[b] > (int64_t(1) << 30)) return BSP_ERR_UNSUPPORTED;
        row_off[b] = static_cast<int32_t>(total_rows);
        total_rows += rows[b];
    }
    const int32_t* prefix_len = pl.data();
    const int32_t* tail_len = tl.data();

    int max_p = 0, max_total = 0, max_t = 0;
    int64_t total_pages = 0;
    for (int b = 0; b < batch; ++b) {
        if (prefix_len[b] < 0 || tail_len[b] < 0) return BSP_ERR_INVALID_ARG;
        if (prefix_len[b] > (1 << 30)) return BSP_ERR_UNSUPPORTED;
        if (tail_len[b] > max_tail) return BSP_ERR_CAPACITY;
        max_p = std::max(max_p, prefix_len[b]);
        max_total = std::max(max_total, prefix_len[b] + tail_len[b]);
        max_t = std::max(max_t, tail_len[b]);
        total_pages += ceil_div(prefix_len[b], ps);
    }
    if (max_p > 0) {
        if (!prefix_pages) return BSP_ERR_INVALID_ARG;
        if (ceil_div(max_p, ps) > prefix_pages_stride) return BSP_ERR_INVALID_ARG;
    }
    for (int b = 0; b < batch; ++b) {
        const int64_t n = ceil_div(prefix_len[b], ps);
        for (int64_t j = 0; j < n; ++j) {
            const int32_t pg = prefix_pages[static_cast<int64_t>(b) * prefix_pages_stride + j];
            if (pg < 0 || pg >= geo->num_pages) return BSP_ERR_PAGE_INDEX;
        }
    }

    // ---- work units: (request, kv head, key split, query-row block)
    int nrb, wblk;
    // prompt tokens per unit of a prefill: one MMA block of rows, or at head_dim <= 128 two of them (the
    // two-block kernel, layout 2: both blocks' rows against the same K/V tiles)
    int urows = 0;
    if (pf) {
        // prompt tokens in blocks of one MMA's rows: 128 / G tokens (dense layout), or at head_dim <= 128
        // 4 * floor(32 / G) tokens, 32 / G per TMEM lane quadrant, two blocks per unit
        const bool two = geo->head_dim <= 128;
        wblk = two ? 4 * (32 / G) : std::max(1, kRowsPerBlock / G);
        urows = two ? 2 * wblk : wblk;
        nrb = 0;
        for (int b = 0; b < batch; ++b) nrb = std::max<int>(nrb, static_cast<int>(ceil_div(rows[b], urows)));
    } else {
        row_blocks(beam_width, G, &nrb, &wblk);
    }
    // The prompt kernel of a decode step at head_dim <= 128 (prefill and head_dim 256: the one-set
    // kernel, layout 0). A row block of at most 64 query rows, 16 per TMEM lane quadrant, keeps the one-set
    // kernel's half-row layout (two threads per row). Otherwise a (request, kv head) with 129-256 rows
    // goes to the wide kernel (layout 2: all its rows in one unit as two MMA blocks, the prompt read
    // once), and any other to the alternating-tile kernel (layout 1), whose row blocks of one (request,
    // kv head, key split) are dealt to `group` neighbouring CTAs at the same place of their lists.
    int layout = 0;
    const bool e4m3 = geo->kv_dtype == BSP_KV_DTYPE_E4M3;
    if (e4m3) {
        // E4M3 pools: the wide and alternating-tile kernels widen the tiles (head_dim <= 128, decode); a
        // row block holds at most 4 * floor(32 / G) beams, so that its rows fit the quadrant layout
        if (pf || geo->head_dim > 128) return BSP_ERR_UNSUPPORTED;
        if (wide_quad_beams(geo->head_dim, beam_width, G) > 0) {
            layout = 2;
            nrb = 1;
            wblk = beam_width;
        } else {
            if (alt_quad_beams(geo->head_dim, wblk, G) == 0) {
                const int wmax = 4 * (32 / G);
                nrb = static_cast<int>(ceil_div(beam_width, wmax));
                wblk = static_cast<int>(ceil_div(beam_width, nrb));
            }
            layout = 1;
        }
    } else if (pf) {
        if (geo->head_dim <= 128) layout = 2;
    } else if (geo->head_dim <= 128 && prefix_quad_beams(geo->head_dim, wblk, G) == 0) {
        if (wide_quad_beams(geo->head_dim, beam_width, G) > 0) {
            layout = 2;
            nrb = 1;
            wblk = beam_width;
        } else if (alt_quad_beams(geo->head_dim, wblk, G) > 0) {
            layout = 1;
        }
    }
    const bool alt = layout == 1;
    const int group = alt ? nrb : 1;
    if (!pf) urows = wblk;
    auto nrb_of = [&](int b) -> int { return pf ? static_cast<int>(ceil_div(rows[b], urows)) : nrb; };
    std::vector<int64_t> tiles(batch);
    int64_t total_tiles = 0, active = 0;
    for (int b = 0; b < batch; ++b) {
        tiles[b] = ceil_div(prefix_len[b], kTileKeys);
        total_tiles += tiles[b];
        active += tiles[b] > 0;
    }
    int64_t base_units = 0;
    for (int b = 0; b < batch; ++b) base_units += tiles[b] > 0 ? static_cast<int64_t>(Hkv) * nrb_of(b) : 0;
    const int64_t target = 2 * static_cast<int64_t>(num_sms);
    int64_t chunk = std::numeric_limits<int32_t>::max();  // tiles per split
    if (!pf && base_units > 0 && base_units < target)  // (a prefill's key ranges are chosen below)
        chunk = std::max<int64_t>(2, ceil_div(total_tiles * Hkv * nrb, target));
    std::vector<int32_t> nsplit(batch);
    int64_t parts = 0;
    for (;;) {
        parts = 0;
        for (int b = 0; b < batch; ++b) {
            nsplit[b] = tiles[b] == 0 ? 0 : static_cast<int32_t>(ceil_div(tiles[b], chunk));
            parts += nsplit[b];
        }
        if (parts <= static_cast<int64_t>(batch) + kExtraParts) break;
        chunk *= 2;
    }
    const int tk = prefix_tile_keys(geo->head_dim);
    const int64_t unit_ends = layout == 2 ? 8 : 4;
    // the plan tiles a unit reads: a causal prefill block stops at its last token's keys
    auto unit_end_tile = [&](int b, int rb, int32_t t1) -> int32_t {
        if (causal[b] < 0) return t1;
        const int64_t last_row = std::min<int64_t>(rows[b], static_cast<int64_t>(rb + 1) * urows);
        return static_cast<int32_t>(std::min<int64_t>(t1, ceil_div(causal[b] + last_row, kTileKeys)));
    };
    // key range [t0, t1) of split s of request b, in plan tiles
    std::vector<std::vector<int32_t>> pf_cut(pf ? batch : 0);
    if (pf) {
        // A prefill's units are (request, kv head, row block): a long cached prefix makes a request's
        // units the longest of the launch, and the largest CTA load cannot drop below the longest unit.
        // The cached rows of a request whose longest unit is above twice the mean CTA load are cut into
        // about longest / mean key ranges of equal length, each cut inside the cached rows so that every
        // row of every block has keys in every range (the last range holds the rest and the prompt),
        // while the extra partial states last. Below twice the mean the fp32 partial states and the
        // merge cost more than the balance gains. Costs as the dealing below counts them: eighths of a
        // kernel tile.
        auto full_cost = [&](int b, int rb) -> int64_t {
            const int64_t keys = std::min<int64_t>(static_cast<int64_t>(unit_end_tile(b, rb, static_cast<int32_t>(tiles[b]))) *
                                                       kTileKeys, prefix_len[b]);
            return 8 * ceil_div(keys, tk) + unit_ends;
        };
        int64_t total = 0;
        std::vector<int> order;
        for (int b = 0; b < batch; ++b) {
            if (tiles[b] == 0) continue;
            order.push_back(b);
            for (int rb = 0; rb < nrb_of(b); ++rb) total += static_cast<int64_t>(Hkv) * full_cost(b, rb);
        }
        const int64_t mean = std::max<int64_t>(1, ceil_div(total, num_sms));
        std::stable_sort(order.begin(), order.end(), [&](int a, int c) {
            return full_cost(a, nrb_of(a) - 1) > full_cost(c, nrb_of(c) - 1);
        });
        int64_t extra = 0;
        for (int b = 0; b < batch; ++b) pf_cut[b] = {0, static_cast<int32_t>(tiles[b])};
        for (int b : order) {
            const int64_t longest = full_cost(b, nrb_of(b) - 1);
            int64_t n = pf->splits && longest > 2 * mean ? ceil_div(longest, mean) : 1;
            n = std::min<int64_t>(n, 1 + kExtraParts - extra);
            const int32_t span = unit_end_tile(b, nrb_of(b) - 1, static_cast<int32_t>(tiles[b]));
            const int32_t cmax = pf->cached_len[b] / kTileKeys;  // cuts at or below the cached rows
            for (; n > 1; --n) {
                std::vector<int32_t> cut{0};
                bool okc = true;
                for (int64_t i = 1; i < n && okc; ++i) {
                    const int32_t c = std::min<int32_t>(static_cast<int32_t>(i * span / n), cmax);
                    okc = c > cut.back();
                    cut.push_back(c);
                }
                if (!okc) continue;
                cut.push_back(static_cast<int32_t>(tiles[b]));
                pf_cut[b] = cut;
                break;
            }
            nsplit[b] = static_cast<int32_t>(pf_cut[b].size()) - 1;
            extra += nsplit[b] - 1;
        }
        parts = 0;
        for (int b = 0; b < batch; ++b) parts += nsplit[b];
    }
    auto split_range = [&](int b, int s) -> std::pair<int32_t, int32_t> {
        if (pf) return {pf_cut[b][static_cast<size_t>(s)], pf_cut[b][static_cast<size_t>(s) + 1]};
        return {static_cast<int32_t>(s * tiles[b] / nsplit[b]), static_cast<int32_t>((s + 1) * tiles[b] / nsplit[b])};
    };
    auto tail_tiles = [&](int b) -> int64_t { return request_tail_tiles(layout, geo->head_dim, wblk, tail_len[b]); };
    auto fused = [&](int b) -> bool { return request_fused(layout, geo->head_dim, wblk, nsplit[b], tail_len[b]); };
    struct Unit {
        int32_t f[kUnitFields];
    };
    // time of a unit on the prompt kernel, in eighths of a key tile: its TK-key tiles (the last one
    // partial, costed in full), its tail tiles, and the unit's start and end: half a tile, a whole one
    // on the two-block kernel (its units write 256 output rows; measured there as about one tile)
    auto unit_cost = [&](int b, int32_t t0, int32_t t1) -> int64_t {
        const int64_t keys = std::min<int64_t>(static_cast<int64_t>(t1) * kTileKeys, prefix_len[b]) -
                             static_cast<int64_t>(t0) * kTileKeys;
        const int64_t kt = ceil_div(keys, tk) + (fused(b) ? tail_tiles(b) : 0);
        return 8 * kt + unit_ends;
    };
    std::vector<Unit> units;
    units.reserve(static_cast<size_t>(base_units + parts * Hkv * nrb));
    std::vector<int32_t> part_off(batch), page_off(batch);
    int64_t poff = 0, pgoff = 0;
    for (int b = 0; b < batch; ++b) {
        part_off[b] = static_cast<int32_t>(poff);
        page_off[b] = static_cast<int32_t>(pgoff);
        for (int s = 0; s < nsplit[b]; ++s) {
            const auto [t0, t1] = split_range(b, s);
            for (int g = 0; g < Hkv; ++g)
                for (int rb = 0; rb < (group > 1 ? 1 : nrb_of(b)); ++rb) {  // a group's other blocks follow
                    const int32_t te = unit_end_tile(b, rb, t1);
                    Unit u{};
                    u.f[kUnitReq] = b;
                    u.f[kUnitKvHead] = g;
                    u.f[kUnitRowBlock] = rb;
                    u.f[kUnitTile0] = t0;
                    u.f[kUnitTile1] = te;
                    u.f[kUnitPart] = static_cast<int32_t>(poff + s);
                    u.f[kUnitCost] = static_cast<int32_t>(unit_cost(b, t0, te));
                    units.push_back(u);
                }
        }
        poff += nsplit[b];
        pgoff += ceil_div(prefix_len[b], ps);
    }
    // Units go to the persistent CTAs so that the largest per-CTA cost (unit_cost) is small.
    // Longest units first (row blocks of one split stay adjacent: equal keys keep their
    // order); LPT (each unit to the least-loaded CTA) gives an upper bound L on the largest
    // load, then MULTIFIT (Coffman, Garey & Johnson 1978) looks for the smallest capacity
    // C < L at which first-fit-decreasing packs every unit into at most num_sms bins. With
    // few units per CTA, LPT alone can stack four short units on one CTA while others hold
    // three long ones. The list is written grouped by CTA; cta_off[c] .. cta_off[c+1] are
    // CTA c's units, longest first.
    if (units.size() > static_cast<size_t>(std::numeric_limits<int32_t>::max())) return BSP_ERR_UNSUPPORTED;
    {
        // stable: by cost, then by creation order
        std::vector<std::pair<int64_t, int32_t>> key(units.size());
        for (size_t i = 0; i < units.size(); ++i) key[i] = {-static_cast<int64_t>(units[i].f[kUnitCost]), static_cast<int32_t>(i)};
        std::sort(key.begin(), key.end());
        std::vector<Unit> sorted(units.size());
        for (size_t i = 0; i < units.size(); ++i) sorted[i] = units[static_cast<size_t>(key[i].second)];
        units.swap(sorted);
    }
    const int64_t nu = static_cast<int64_t>(units.size());
    auto utiles = [&](int64_t i) -> int64_t { return units[i].f[kUnitCost]; };
    std::vector<std::vector<int32_t>> lists;
    if (nu > 0) {
        const int64_t bins = std::min<int64_t>(nu, num_sms / group);
        if (bins >= (int64_t{1} << 20)) return BSP_ERR_UNSUPPORTED;
        // LPT: a binary min-heap of (load << 20 | cta) keys, ties to the lower CTA index
        std::vector<uint64_t> heap(static_cast<size_t>(bins));
        for (int64_t c = 0; c < bins; ++c) heap[static_cast<size_t>(c)] = static_cast<uint64_t>(c);  // a heap already
        int64_t total = 0, lpt_max = 0;
        std::vector<int32_t> lpt_assign(static_cast<size_t>(nu));
        for (int64_t i = 0; i < nu; ++i) {
            const uint64_t top = heap[0];
            const int64_t c = static_cast<int64_t>(top & 0xFFFFFu);
            const int64_t ld = static_cast<int64_t>(top >> 20) + utiles(i);
            lpt_assign[static_cast<size_t>(i)] = static_cast<int32_t>(c);
            lpt_max = std::max(lpt_max, ld);
            total += utiles(i);
            // replace the root with the grown load and sift it down
            const uint64_t key = (static_cast<uint64_t>(ld) << 20) | static_cast<uint64_t>(c);
            size_t pos = 0;
            const size_t n = heap.size();
            for (;;) {
                size_t ch = 2 * pos + 1;
                if (ch >= n) break;
                if (ch + 1 < n && heap[ch + 1] < heap[ch]) ++ch;
                if (heap[ch] >= key) break;
                heap[pos] = heap[ch];
                pos = ch;
            }
            heap[pos] = key;
        }
        // first-fit-decreasing into `bins` bins of capacity cap (false if a unit fits none): each unit
        // goes to the lowest-numbered bin with room, found in a max-tree of the bins' free capacity,
        // so a probe costs O(units x log bins); the same packing as opening bins one by one
        int64_t tsize = 1;
        while (tsize < bins) tsize <<= 1;
        std::vector<int64_t> tree(static_cast<size_t>(2 * tsize));
        std::vector<int32_t> assign(static_cast<size_t>(nu)), best_assign;
        auto pack = [&](int64_t cap) -> bool {
            for (int64_t j = 0; j < tsize; ++j) tree[static_cast<size_t>(tsize + j)] = j < bins ? cap : -1;
            for (int64_t v = tsize - 1; v >= 1; --v)
                tree[static_cast<size_t>(v)] = std::max(tree[static_cast<size_t>(2 * v)], tree[static_cast<size_t>(2 * v + 1)]);
            for (int64_t i = 0; i < nu; ++i) {
                const int64_t x = utiles(i);
                if (tree[1] < x) return false;
                int64_t v = 1;
                while (v < tsize) v = tree[static_cast<size_t>(2 * v)] >= x ? 2 * v : 2 * v + 1;
                assign[static_cast<size_t>(i)] = static_cast<int32_t>(v - tsize);
                tree[static_cast<size_t>(v)] -= x;
                for (v >>= 1; v >= 1; v >>= 1)
                    tree[static_cast<size_t>(v)] =
                        std::max(tree[static_cast<size_t>(2 * v)], tree[static_cast<size_t>(2 * v + 1)]);
            }
            return true;
        };
        // the smallest capacity below LPT's largest load at which FFD packs, by bisection; a packing
        // that succeeds bounds the answer by its own largest load, which may be below the probe
        int64_t lo = std::max<int64_t>(ceil_div(total, bins), utiles(0)), hi = lpt_max - 1;
        while (lo <= hi) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (pack(mid)) {
                best_assign = assign;
                int64_t used = 0;  // the packing's largest load: cap minus the least free capacity
                for (int64_t j = 0; j < bins; ++j)
                    used = std::max(used, mid - tree[static_cast<size_t>(tsize + j)]);
                hi = std::min(mid, used) - 1;
            } else {
                lo = mid + 1;
            }
        }
        // the CTAs' unit lists from MULTIFIT's packing, or LPT's when no smaller capacity packs
        {
            const std::vector<int32_t>& a = best_assign.empty() ? lpt_assign : best_assign;
            std::vector<int32_t> cnt(static_cast<size_t>(bins), 0);
            for (int64_t i = 0; i < nu; ++i) ++cnt[static_cast<size_t>(a[static_cast<size_t>(i)])];
            lists.assign(static_cast<size_t>(bins), {});
            for (int64_t c = 0; c < bins; ++c) lists[static_cast<size_t>(c)].reserve(static_cast<size_t>(cnt[static_cast<size_t>(c)]) + 2);
            for (int64_t i = 0; i < nu; ++i) lists[static_cast<size_t>(a[static_cast<size_t>(i)])].push_back(static_cast<int32_t>(i));
        }
        // local search on the most-loaded CTA: move one of its units to a CTA that stays below
        // its load, or swap one of its units for a shorter one of another CTA; stop when
        // neither lowers it
        std::vector<int64_t> load(static_cast<size_t>(bins), 0);
        for (int64_t c = 0; c < bins; ++c)
            for (int32_t i : lists[static_cast<size_t>(c)]) load[static_cast<size_t>(c)] += utiles(i);
        for (int iter = 0; iter < 4 * nu; ++iter) {
            const size_t a = static_cast<size_t>(std::max_element(load.begin(), load.end()) - load.begin());
            const int64_t M = load[a];
            bool moved = false;
            for (size_t xi = 0; xi < lists[a].size() && !moved; ++xi) {
                const int64_t x = utiles(lists[a][xi]);
                for (size_t b = 0; b < load.size() && !moved; ++b) {
                    if (b == a) continue;
                    if (load[b] + x < M) {
                        lists[b].push_back(lists[a][xi]);
                        lists[a].erase(lists[a].begin() + static_cast<std::ptrdiff_t>(xi));
                        load[b] += x;
                        load[a] -= x;
                        moved = true;
                        break;
                    }
                    for (size_t yi = 0; yi < lists[b].size(); ++yi) {
                        const int64_t y = utiles(lists[b][yi]);
                        if (y < x && load[b] - y + x < M) {
                            std::swap(lists[a][xi], lists[b][yi]);
                            load[a] += y - x;
                            load[b] += x - y;
                            moved = true;
                            break;
                        }
                    }
                }
            }
            if (!moved) break;
        }
        lists.erase(std::remove_if(lists.begin(), lists.end(), [](const std::vector<int32_t>& l) { return l.empty(); }),
                    lists.end());
        for (auto& l : lists)  // longest first within a CTA (stable insertion sort: a few units each)
            for (size_t i = 1; i < l.size(); ++i) {
                const int32_t x = l[i];
                size_t j = i;
                while (j > 0 && utiles(l[j - 1]) < utiles(x)) {
                    l[j] = l[j - 1];
                    --j;
                }
                l[j] = x;
            }
        if (group > 1) {
            // each dealt list goes to `group` neighbouring CTAs, one per row block, in the same order
            std::vector<Unit> all;
            std::vector<std::vector<int32_t>> glists;
            all.reserve(units.size() * static_cast<size_t>(group));
            for (const auto& l : lists)
                for (int rb = 0; rb < group; ++rb) {
                    glists.emplace_back();
                    for (int32_t i : l) {
                        Unit u = units[static_cast<size_t>(i)];
                        u.f[kUnitRowBlock] = rb;
                        glists.back().push_back(static_cast<int32_t>(all.size()));
                        all.push_back(u);
                    }
                }
            units.swap(all);
            lists.swap(glists);
        }
    }
    const int64_t ctas = static_cast<int64_t>(lists.size());
    // a decode plan's CTA table has num_sms + 1 entries (CTAs past `ctas` have no units), so a launch
    // of num_sms CTAs captured in a CUDA graph reads a valid table after any later plan
    const bool fixed = !pf && fixed_layout;
    std::vector<int32_t> cta_off(static_cast<size_t>(fixed ? std::max<int64_t>(ctas, num_sms) : ctas) + 1, 0);
    {
        std::vector<Unit> dealt;
        dealt.reserve(units.size());
        for (int64_t c = 0; c < ctas; ++c) {
            for (int32_t i : lists[static_cast<size_t>(c)]) dealt.push_back(units[i]);
            cta_off[static_cast<size_t>(c) + 1] = static_cast<int32_t>(dealt.size());
        }
        for (size_t c = static_cast<size_t>(ctas) + 1; c < cta_off.size(); ++c) cta_off[c] = static_cast<int32_t>(dealt.size());
        units.swap(dealt);
    }

    // ---- image. A decode plan has a fixed layout for its batch, beam width, SM count and page-table
    // stride: every section at an offset that does not depend on the lengths (the unit list sized
    // for the most key splits the planner makes), so the device addresses baked into a captured
    // CUDA graph stay valid for every later plan of the same shape. A prefill plan is packed.
    const int64_t parts_cap = fixed ? static_cast<int64_t>(batch) + kExtraParts : parts;
    // rows of a request's partial-state slot: the beams of a decode step, the longest prompt of a prefill
    // with key splits (a prefill without them writes no partial state)
    int32_t part_w = beam_width;
    if (pf && std::any_of(nsplit.begin(), nsplit.end(), [](int32_t n) { return n > 1; }))
        for (int b = 0; b < batch; ++b) part_w = std::max(part_w, rows[b]);
    const size_t units_cap = fixed ? static_cast<size_t>(parts_cap) * Hkv * nrb : units.size();
    const size_t pages_cap = fixed ? static_cast<size_t>(batch) * prefix_pages_stride : static_cast<size_t>(total_pages);
    if (units.size() > units_cap || static_cast<size_t>(total_pages) > pages_cap) return BSP_ERR_CAPACITY;
    const size_t off_req = kImageHeaderBytes;
    const size_t off_units = off_req + static_cast<size_t>(batch) * kReqFields * 4;
    const size_t off_cta = off_units + units_cap * kUnitFields * 4;
    const size_t off_pages = off_cta + cta_off.size() * 4;
    const size_t need = off_pages + pages_cap * 4;
    if (!image || image_bytes < need) return BSP_ERR_CAPACITY;
    uint8_t* img = static_cast<uint8_t*>(image);
    std::memset(img, 0, kImageHeaderBytes);
    // header: [2] batch, [3] units, [4] beam width, [5] SM count, [6] kind, [7] tail bound (what a
    // replayed graph checks against its capture)
    reinterpret_cast<int32_t*>(img)[2] = batch;
    reinterpret_cast<int32_t*>(img)[3] = static_cast<int32_t>(units.size());
    reinterpret_cast<int32_t*>(img)[4] = part_w;
    reinterpret_cast<int32_t*>(img)[5] = num_sms;
    reinterpret_cast<int32_t*>(img)[6] = pf ? 1 : 0;
    reinterpret_cast<int32_t*>(img)[7] = max_tail;
    int32_t* req = reinterpret_cast<int32_t*>(img + off_req);
    for (int b = 0; b < batch; ++b) {
        int32_t* r = req + static_cast<size_t>(b) * kReqFields;
        std::memset(r, 0, kReqFields * 4);
        r[kReqPrefix] = prefix_len[b];
        r[kReqTail] = tail_len[b];
        r[kReqSplits] = nsplit[b];
        r[kReqPartOff] = part_off[b];
        r[kReqPageOff] = page_off[b];
        r[kReqFused] = fused(b) ? 1 : 0;
        r[kReqRows] = rows[b];
        r[kReqCausal] = causal[b];
        r[kReqRowOff] = row_off[b];
    }
    if (!units.empty()) std::memcpy(img + off_units, units.data(), units.size() * sizeof(Unit));
    std::memcpy(img + off_cta, cta_off.data(), cta_off.size() * 4);
    int32_t* pages = reinterpret_cast<int32_t*>(img + off_pages);
    for (int b = 0; b < batch; ++b) {
        const int64_t n = ceil_div(prefix_len[b], ps);
        if (n) std::memcpy(pages + page_off[b], prefix_pages + static_cast<int64_t>(b) * prefix_pages_stride, n * 4);
    }

    std::memset(out, 0, sizeof(*out));
    out->geo = *geo;
    out->batch = batch;
    out->beam_width = part_w;
    out->max_tail = max_tail;
    out->prefix_pages_stride = prefix_pages_stride;
    out->num_units = static_cast<int32_t>(units.size());
    out->num_parts = static_cast<int32_t>(parts);
    out->row_blocks = nrb;
    out->beams_per_block = wblk;
    out->tile_keys = kTileKeys;
    out->max_prefix_len = max_p;
    out->max_total_len = max_total;
    out->num_sms = num_sms;
    out->max_tail_len = max_t;
    out->prefix_ctas = static_cast<int32_t>(ctas);
    int32_t tail_requests = 0;
    // (a prefill request is the tail kernel's when its keys were split)
    for (int b = 0; b < batch; ++b) tail_requests += pf ? nsplit[b] > 1 : !fused(b);
    out->tail_requests = tail_requests;
    out->total_rows = static_cast<int32_t>(total_rows);
    out->kind = pf ? 1 : 0;
    out->layout = layout;
    out->image_bytes = need;
    // offsets relative to the device workspace
    DeviceLayout L = device_layout(need, parts_cap, part_w, *geo);
    out->off_req = kStatusBytes + off_req;
    out->off_units = kStatusBytes + off_units;
    out->off_cta = kStatusBytes + off_cta;
    out->off_pages = kStatusBytes + off_pages;
    out->off_part_lse = kStatusBytes + L.image;
    out->off_part_o = kStatusBytes + L.image + L.part_lse;
    out->device_bytes_used = L.total;
    return BSP_OK;
}
}  // namespace

extern "C" {

bsp_status bsp_plan_build(const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len,
                          const int32_t* tail_len, const int32_t* prefix_pages, int32_t prefix_pages_stride,
                          int32_t max_tail, int32_t num_sms, void* image, size_t image_bytes, bsp_plan_t* out) {
    return plan_build_core(geo, batch, beam_width, prefix_len, tail_len, prefix_pages, prefix_pages_stride, max_tail,
                           num_sms, image, image_bytes, out, nullptr);
}

}  // extern "C"

namespace bsp {
// A decode plan with the packed layout (sections and partial states sized by this plan's own units and
// splits), for a caller that never replays it from a CUDA graph: the fixed-scratch entry point.
bsp_status plan_build_packed(const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len,
                             const int32_t* tail_len, const int32_t* prefix_pages, int32_t prefix_pages_stride,
                             int32_t max_tail, int32_t num_sms, void* image, size_t image_bytes, bsp_plan_t* out) {
    return plan_build_core(geo, batch, beam_width, prefix_len, tail_len, prefix_pages, prefix_pages_stride, max_tail,
                           num_sms, image, image_bytes, out, nullptr, false);
}
}  // namespace bsp

extern "C" {

bsp_status bsp_plan_prefill_build(const bsp_geometry* geo, int32_t batch, const int32_t* cached_len,
                                  const int32_t* prompt_len, const int32_t* pages, int32_t pages_stride,
                                  int32_t causal, int32_t num_sms, void* image, size_t image_bytes,
                                  bsp_plan_t* out) {
    const PrefillSpec pf{cached_len, prompt_len, causal != 0, true};
    return plan_build_core(geo, batch, 1, nullptr, nullptr, pages, pages_stride, 0, num_sms, image, image_bytes, out,
                           &pf);
}

}  // extern "C"

namespace {
// The staging slot of generation `gen` (slot gen & 1), once the stream has executed the copy that last
// read it (generation gen - 2, echoed back into the header); waits up to 10 s.
bsp_status acquire_slot(StagingHeader* hdr, uint64_t gen, cudaStream_t s, uint8_t** slot_ptr) {
    const int slot = static_cast<int>(gen & 1);
    *slot_ptr = reinterpret_cast<uint8_t*>(hdr) + kStagingHeaderBytes + slot * hdr->slot_bytes;
    if (gen >= 3) {
        const auto t0 = std::chrono::steady_clock::now();
        while (reinterpret_cast<volatile uint64_t*>(hdr->echoed)[slot] < gen - 2) {
            cudaError_t q = cudaStreamQuery(s);
            if (q != cudaSuccess && q != cudaErrorNotReady) return BSP_ERR_CUDA;
            if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10)) return BSP_ERR_CUDA;
            std::this_thread::yield();
        }
    }
    return BSP_OK;
}

// Stamps generation `gen` into the image in `slot_ptr`, enqueues the copy of its first `bytes` bytes into
// the device workspace and the echo of the generation back into the header, and makes `gen` current.
bsp_status enqueue_image(StagingHeader* hdr, uint64_t gen, uint8_t* slot_ptr, size_t bytes, void* ws_device,
                         cudaStream_t s) {
    std::memcpy(slot_ptr, &gen, sizeof gen);  // image header: generation
    uint8_t* dimg = static_cast<uint8_t*>(ws_device) + kStatusBytes;
    if (cudaMemcpyAsync(dimg, slot_ptr, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return BSP_ERR_CUDA;
    if (cudaMemcpyAsync(&hdr->echoed[gen & 1], dimg, sizeof(uint64_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    hdr->generation = gen;
    return BSP_OK;
}

// Builds a plan into a free slot of the pinned staging buffer (build(sms, slot, bytes, plan)) and
// enqueues its copy into the device workspace with the generation echo.
template <typename Build>
bsp_status stage_plan(void* ws_device, size_t ws_device_bytes, void* ws_host, size_t ws_host_bytes, void* stream,
                      bsp_plan_t* out, Build build) {
    if (!out || !ws_device || !ws_host) return BSP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws_device) & (kAlign - 1)) || (reinterpret_cast<uintptr_t>(ws_host) & 63u))
        return BSP_ERR_INVALID_ARG;
    if (ws_host_bytes < kStagingHeaderBytes + 2 * kAlign) return BSP_ERR_CAPACITY;
    if (ws_device_bytes < kStatusBytes + kAlign) return BSP_ERR_CAPACITY;
    if (!device_ptr_ok(ws_device)) return BSP_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BSP_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    StagingHeader* hdr = static_cast<StagingHeader*>(ws_host);
    if (hdr->magic != kStagingMagic || hdr->ws_device != reinterpret_cast<uint64_t>(ws_device)) {
        std::memset(hdr, 0, kStagingHeaderBytes);
        hdr->magic = kStagingMagic;
        hdr->ws_device = reinterpret_cast<uint64_t>(ws_device);
    }
    const uint64_t gen = hdr->generation + 1;
    hdr->slot_bytes = (ws_host_bytes - kStagingHeaderBytes) / 2 / kAlign * kAlign;
    uint8_t* slot_ptr = nullptr;
    bsp_status st = acquire_slot(hdr, gen, s, &slot_ptr);
    if (st != BSP_OK) return st;
    bsp_plan_t plan;
    st = build(sms, slot_ptr, hdr->slot_bytes, &plan);
    if (st != BSP_OK) return st;
    if (plan.device_bytes_used > ws_device_bytes) return BSP_ERR_CAPACITY;
    st = enqueue_image(hdr, gen, slot_ptr, plan.image_bytes, ws_device, s);
    if (st != BSP_OK) return st;
    plan.generation = gen;
    plan.ws_device = ws_device;
    plan.ws_device_bytes = ws_device_bytes;
    plan.ws_host = ws_host;
    *out = plan;
    return BSP_OK;
}
}  // namespace

extern "C" {

bsp_status bsp_plan(const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len,
                    const int32_t* tail_len, const int32_t* prefix_pages, int32_t prefix_pages_stride, int32_t max_tail,
                    void* ws_device, size_t ws_device_bytes, void* ws_host, size_t ws_host_bytes, void* stream,
                    bsp_plan_t* out) {
    return stage_plan(ws_device, ws_device_bytes, ws_host, ws_host_bytes, stream, out,
                      [&](int sms, void* img, size_t bytes, bsp_plan_t* p) {
                          return bsp_plan_build(geo, batch, beam_width, prefix_len, tail_len, prefix_pages,
                                                prefix_pages_stride, max_tail, sms, img, bytes, p);
                      });
}

bsp_status bsp_plan_prefill(const bsp_geometry* geo, int32_t batch, const int32_t* cached_len,
                            const int32_t* prompt_len, const int32_t* pages, int32_t pages_stride, int32_t causal,
                            void* ws_device, size_t ws_device_bytes, void* ws_host, size_t ws_host_bytes, void* stream,
                            bsp_plan_t* out) {
    return stage_plan(ws_device, ws_device_bytes, ws_host, ws_host_bytes, stream, out,
                      [&](int sms, void* img, size_t bytes, bsp_plan_t* p) {
                          bsp_status r = bsp_plan_prefill_build(geo, batch, cached_len, prompt_len, pages,
                                                                pages_stride, causal, sms, img, bytes, p);
                          if (r == BSP_OK && p->device_bytes_used > ws_device_bytes) {
                              // no room for the partial states of key splits: the plan without them
                              const PrefillSpec pf{cached_len, prompt_len, causal != 0, false};
                              r = plan_build_core(geo, batch, 1, nullptr, nullptr, pages, pages_stride, 0, sms, img,
                                                  bytes, p, &pf);
                          }
                          return r;
                      });
}

bsp_status bsp_plan_update_tails(bsp_plan_t* plan, const int32_t* tail_len, void* stream) {
    bsp_status st = check_plan(plan);
    if (st != BSP_OK) return st;
    if (plan->kind != 0) return BSP_ERR_INVALID_ARG;
    const int B = plan->batch;
    if (B > 0 && !tail_len) return BSP_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b) {
        if (tail_len[b] < 0) return BSP_ERR_INVALID_ARG;
        if (tail_len[b] > plan->max_tail) return BSP_ERR_CAPACITY;
    }
    StagingHeader* hdr = static_cast<StagingHeader*>(plan->ws_host);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the current image (header and request records) is in the current generation's slot
    const uint8_t* cur = reinterpret_cast<const uint8_t*>(hdr) + kStagingHeaderBytes + (hdr->generation & 1) * hdr->slot_bytes;
    const uint64_t gen = hdr->generation + 1;
    uint8_t* slot_ptr = nullptr;
    st = acquire_slot(hdr, gen, s, &slot_ptr);
    if (st != BSP_OK) return st;
    const size_t bytes = plan->off_units - kStatusBytes;  // the image header and the request records
    std::memcpy(slot_ptr, cur, bytes);
    int32_t* req = reinterpret_cast<int32_t*>(slot_ptr + (plan->off_req - kStatusBytes));
    int32_t max_t = 0, max_total = 0, tail_requests = 0;
    for (int b = 0; b < B; ++b) {
        int32_t* r = req + static_cast<size_t>(b) * kReqFields;
        r[kReqTail] = tail_len[b];
        r[kReqFused] = request_fused(plan->layout, plan->geo.head_dim, plan->beams_per_block, r[kReqSplits], tail_len[b]);
        tail_requests += !r[kReqFused];
        max_t = std::max(max_t, tail_len[b]);
        max_total = std::max(max_total, r[kReqPrefix] + tail_len[b]);
    }
    st = enqueue_image(hdr, gen, slot_ptr, bytes, plan->ws_device, s);
    if (st != BSP_OK) return st;
    plan->generation = gen;
    plan->max_tail_len = max_t;
    plan->max_total_len = max_total;
    plan->tail_requests = tail_requests;
    return BSP_OK;
}

bsp_status bsp_append_kv(const bsp_plan_t* plan, const void* k_new, const void* v_new, int64_t src_row_stride,
                         const int32_t* out_cache_loc, int32_t n, void* k_pool, void* v_pool,
                         void* const* events, void* stream) {
    bsp_status st = check_plan(plan);
    if (st != BSP_OK) return st;
    if (n < 0 || plan->geo.kv_dtype != BSP_KV_DTYPE_SAME) return BSP_ERR_INVALID_ARG;  // 16-bit pools only
    if (n == 0) return BSP_OK;
    const bsp_geometry& geo = plan->geo;
    if (n > plan->total_rows) return BSP_ERR_INVALID_ARG;
    if (src_row_stride < static_cast<int64_t>(geo.num_kv_heads) * geo.head_dim || (src_row_stride & 7))
        return BSP_ERR_INVALID_ARG;
    if (!device_ptr_ok(k_new) || !device_ptr_ok(v_new) || !device_ptr_ok(out_cache_loc) || !device_ptr_ok(k_pool) ||
        !device_ptr_ok(v_pool))
        return BSP_ERR_INVALID_ARG;
    AppendParams p{};
    p.k_new = k_new;
    p.v_new = v_new;
    p.src_row_stride = src_row_stride;
    p.loc = out_cache_loc;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.status = static_cast<int32_t*>(plan->ws_device);
    p.n = n;
    p.Hkv = geo.num_kv_heads;
    p.D = geo.head_dim;
    p.ps_log2 = ilog2(geo.page_size);
    p.num_pages = geo.num_pages;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (prepare_append() != cudaSuccess) return BSP_ERR_CUDA;
    if (!record_event(events, 0, s)) return BSP_ERR_CUDA;
    if (launch_append(p, s) != cudaSuccess) return BSP_ERR_CUDA;
    return record_event(events, 1, s) ? BSP_OK : BSP_ERR_CUDA;
}

bsp_status bsp_append_kv_fp8(const bsp_plan_t* plan, const void* k_new, const void* v_new, int64_t src_row_stride,
                             int32_t src_dtype, float k_mul, float v_mul, const int32_t* out_cache_loc, int32_t n,
                             void* k_pool, void* v_pool, void* const* events, void* stream) {
    bsp_status st = check_plan(plan);
    if (st != BSP_OK) return st;
    if (n < 0) return BSP_ERR_INVALID_ARG;
    if (src_dtype != BSP_FP8_SRC_16BIT && src_dtype != BSP_FP8_SRC_E4M3) return BSP_ERR_INVALID_ARG;
    if (src_dtype == BSP_FP8_SRC_16BIT && (!std::isfinite(k_mul) || !std::isfinite(v_mul) || !(k_mul > 0.f) ||
                                           !(v_mul > 0.f)))
        return BSP_ERR_INVALID_ARG;
    if (n == 0) return BSP_OK;
    const bsp_geometry& geo = plan->geo;
    if (n > plan->total_rows) return BSP_ERR_INVALID_ARG;
    const int64_t align = src_dtype == BSP_FP8_SRC_E4M3 ? 16 : 8;  // elements in 16 bytes
    if (src_row_stride < static_cast<int64_t>(geo.num_kv_heads) * geo.head_dim || (src_row_stride % align))
        return BSP_ERR_INVALID_ARG;
    if (!device_ptr_ok(k_new) || !device_ptr_ok(v_new) || !device_ptr_ok(out_cache_loc) || !device_ptr_ok(k_pool) ||
        !device_ptr_ok(v_pool))
        return BSP_ERR_INVALID_ARG;
    AppendFp8Params p{};
    p.k_new = k_new;
    p.v_new = v_new;
    p.src_row_stride = src_row_stride;
    p.loc = out_cache_loc;
    p.k_pool = static_cast<uint8_t*>(k_pool);
    p.v_pool = static_cast<uint8_t*>(v_pool);
    p.status = static_cast<int32_t*>(plan->ws_device);
    p.k_mul = k_mul;
    p.v_mul = v_mul;
    p.n = n;
    p.Hkv = geo.num_kv_heads;
    p.D = geo.head_dim;
    p.ps_log2 = ilog2(geo.page_size);
    p.num_pages = geo.num_pages;
    // the 16-bit source is the geometry's dtype
    const int src = src_dtype == BSP_FP8_SRC_E4M3 ? 2 : (geo.dtype == BSP_DTYPE_BF16 ? 0 : 1);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (prepare_append_fp8(src) != cudaSuccess) return BSP_ERR_CUDA;
    if (!record_event(events, 0, s)) return BSP_ERR_CUDA;
    if (launch_append_fp8(src, p, s) != cudaSuccess) return BSP_ERR_CUDA;
    return record_event(events, 1, s) ? BSP_OK : BSP_ERR_CUDA;
}

bsp_status bsp_rope_cos_sin(int32_t max_position, int32_t rotary_dim, double base, float* cos_sin, void* stream) {
    if (max_position <= 0 || rotary_dim < 2 || rotary_dim > 1024 || (rotary_dim & 1)) return BSP_ERR_INVALID_ARG;
    if (!(base > 1.0) || !std::isfinite(base)) return BSP_ERR_INVALID_ARG;
    if (!device_ptr_ok(cos_sin)) return BSP_ERR_INVALID_ARG;
    return launch_rope_cos_sin(max_position, rotary_dim, base, cos_sin, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? BSP_OK
               : BSP_ERR_CUDA;
}

static bsp_status rope_append_impl(const bsp_plan_t* plan, const bsp_rope_config* rope, const int32_t* positions,
                                   void* q, int64_t q_row_stride, const void* k_new, const void* v_new,
                                   int64_t src_row_stride, bool fp8, float k_mul, float v_mul,
                                   const int32_t* out_cache_loc, int32_t n, void* k_pool, void* v_pool,
                                   void* const* events, void* stream) {
    bsp_status st = check_plan(plan);
    if (st != BSP_OK) return st;
    if (!rope || n < 0) return BSP_ERR_INVALID_ARG;
    if (!fp8 && plan->geo.kv_dtype != BSP_KV_DTYPE_SAME) return BSP_ERR_INVALID_ARG;  // 16-bit pools only
    if (fp8 && (!std::isfinite(k_mul) || !std::isfinite(v_mul) || !(k_mul > 0.f) || !(v_mul > 0.f)))
        return BSP_ERR_INVALID_ARG;
    const bsp_geometry& geo = plan->geo;
    const int D = geo.head_dim;
    if (rope->rotary_dim < 16 || rope->rotary_dim > D || (rope->rotary_dim & 15) || rope->max_position <= 0 ||
        (rope->interleaved != 0 && rope->interleaved != 1) || rope->reserved != 0)
        return BSP_ERR_INVALID_ARG;
    if (n == 0) return BSP_OK;
    if (n > plan->total_rows) return BSP_ERR_INVALID_ARG;
    if (src_row_stride < static_cast<int64_t>(geo.num_kv_heads) * D || (src_row_stride & 7)) return BSP_ERR_INVALID_ARG;
    if (q && (q_row_stride < static_cast<int64_t>(geo.num_q_heads) * D || (q_row_stride & 7))) return BSP_ERR_INVALID_ARG;
    if (!device_ptr_ok(k_new) || !device_ptr_ok(v_new) || !device_ptr_ok(out_cache_loc) || !device_ptr_ok(positions) ||
        !device_ptr_ok(k_pool) || !device_ptr_ok(v_pool) || !device_ptr_ok(rope->cos_sin) || (q && !device_ptr_ok(q)))
        return BSP_ERR_INVALID_ARG;
    RopeAppendParams p{};
    p.k_new = k_new;
    p.v_new = v_new;
    p.src_row_stride = src_row_stride;
    p.q = q;
    p.q_row_stride = q ? q_row_stride : 0;
    p.loc = out_cache_loc;
    p.pos = positions;
    p.cos_sin = rope->cos_sin;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.status = static_cast<int32_t*>(plan->ws_device);
    p.n = n;
    p.Hq = geo.num_q_heads;
    p.Hkv = geo.num_kv_heads;
    p.ps_log2 = ilog2(geo.page_size);
    p.num_pages = geo.num_pages;
    p.rot = rope->rotary_dim;
    p.interleaved = rope->interleaved;
    p.max_pos = rope->max_position;
    p.k_mul = k_mul;
    p.v_mul = v_mul;
    const bool bf16 = geo.dtype == BSP_DTYPE_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (prepare_rope_append(D, bf16, fp8) != cudaSuccess) return BSP_ERR_CUDA;
    if (!record_event(events, 0, s)) return BSP_ERR_CUDA;
    if (launch_rope_append(D, bf16, fp8, p, s) != cudaSuccess) return BSP_ERR_CUDA;
    return record_event(events, 1, s) ? BSP_OK : BSP_ERR_CUDA;
}

bsp_status bsp_rope_append_kv(const bsp_plan_t* plan, const bsp_rope_config* rope, const int32_t* positions, void* q,
                              int64_t q_row_stride, const void* k_new, const void* v_new, int64_t src_row_stride,
                              const int32_t* out_cache_loc, int32_t n, void* k_pool, void* v_pool,
                              void* const* events, void* stream) {
    return rope_append_impl(plan, rope, positions, q, q_row_stride, k_new, v_new, src_row_stride, false, 1.f, 1.f,
                            out_cache_loc, n, k_pool, v_pool, events, stream);
}

bsp_status bsp_rope_append_kv_fp8(const bsp_plan_t* plan, const bsp_rope_config* rope, const int32_t* positions,
                                  void* q, int64_t q_row_stride, const void* k_new, const void* v_new,
                                  int64_t src_row_stride, float k_mul, float v_mul, const int32_t* out_cache_loc,
                                  int32_t n, void* k_pool, void* v_pool, void* const* events, void* stream) {
    return rope_append_impl(plan, rope, positions, q, q_row_stride, k_new, v_new, src_row_stride, true, k_mul, v_mul,
                            out_cache_loc, n, k_pool, v_pool, events, stream);
}

bsp_status bsp_read_device_status(const bsp_plan_t* plan, void* stream, int32_t clear, int32_t* flags_out) {
    if (!plan || !plan->ws_device) return BSP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return BSP_ERR_CUDA;
    int32_t flags = 0;
    if (cudaMemcpy(&flags, plan->ws_device, sizeof flags, cudaMemcpyDeviceToHost) != cudaSuccess) return BSP_ERR_CUDA;
    if (clear && cudaMemset(plan->ws_device, 0, sizeof flags) != cudaSuccess) return BSP_ERR_CUDA;
    if (flags_out) *flags_out = flags;
    if (flags & (BSP_DEVFLAG_PAGE_INDEX | BSP_DEVFLAG_POSITION)) return BSP_ERR_PAGE_INDEX;
    if (flags & BSP_DEVFLAG_GRAPH) return BSP_ERR_STALE_PLAN;
    if (flags & BSP_DEVFLAG_TIMEOUT) return BSP_ERR_DEVICE_TIMEOUT;
    return BSP_OK;
}

}  // extern "C"

namespace bsp {
// Host-checkable arguments of the attention launches of `plan` (prefill == false: a decode plan, else a
// prefill plan). Nothing is enqueued.
bsp_status attn_check_args(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
                           int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse, bool prefill,
                           bool fp8, float k_scale, float v_scale) {
    if (plan->kind != (prefill ? 1 : 0)) return BSP_ERR_INVALID_ARG;
    if ((plan->geo.kv_dtype == BSP_KV_DTYPE_E4M3) != fp8) return BSP_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !std::isfinite(k_scale) || !(v_scale > 0.f) || !std::isfinite(v_scale))
        return BSP_ERR_INVALID_ARG;
    if (flags & ~(BSP_FLAG_LSE_BASE2 | BSP_FLAG_CHECK | BSP_FLAG_GRAPH)) return BSP_ERR_INVALID_ARG;
    // graph mode: launch shapes that do not depend on the plan's lengths (decode plans only)
    const bool graph = (flags & BSP_FLAG_GRAPH) != 0;
    if (graph && (prefill || (flags & BSP_FLAG_CHECK))) return BSP_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BSP_ERR_INVALID_ARG;
    const bsp_geometry& geo = plan->geo;
    if (plan->total_rows == 0) return BSP_OK;
    if (!device_ptr_ok(q) || !device_ptr_ok(k_pool) || !device_ptr_ok(v_pool) || !device_ptr_ok(o) ||
        !device_ptr_ok(lse))
        return BSP_ERR_INVALID_ARG;
    if (plan->max_tail_len > 0) {
        if (!device_ptr_ok(beam_pages) || !device_ptr_ok(cache_indirection)) return BSP_ERR_INVALID_ARG;
        if (max_seq < plan->max_total_len || max_seq < 1) return BSP_ERR_INVALID_ARG;
        if (beam_pages_stride < ceil_div(plan->max_total_len, geo.page_size)) return BSP_ERR_INVALID_ARG;
    }
    return BSP_OK;
}

// The attention launches of a decode step (prefill == false: the prompt kernel, one or two MMA blocks
// per unit as the plan says, then the tail kernel for the requests that need it) or of a prefill (the
// prompt kernel alone, dense row layout), for a plan whose status word, image and partial states sit
// at `ws`. The arguments have passed attn_check_args.
bsp_status attn_launches(const bsp_plan_t* plan, uint8_t* ws, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
                         int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse,
                         void* const* events, cudaStream_t s, bool prefill, float k_scale, float v_scale) {
    const bool graph = (flags & BSP_FLAG_GRAPH) != 0;
    const bsp_geometry& geo = plan->geo;
    const int64_t R = plan->total_rows;
    if (R == 0) return BSP_OK;
    const int D = geo.head_dim, Hq = geo.num_q_heads, Hkv = geo.num_kv_heads, G = Hq / Hkv;
    const bool bf16 = geo.dtype == BSP_DTYPE_BF16;
    const float log2e = 1.4426950408889634f;
    const bool alt = plan->layout == 1, wide = plan->layout == 2;
    const bool fp8 = geo.kv_dtype == BSP_KV_DTYPE_E4M3;  // the planner gave such a plan layout 1 or 2
    if (fp8 && !alt && !wide) return BSP_ERR_INVALID_ARG;

    // everything that is not a launch (attributes, tensor maps, parameters) comes before the
    // first timing event
    const bool prefix = graph || plan->num_units > 0;
    if (prefix && (alt ? prepare_alt(D, bf16, fp8) : wide ? prepare_wide(D, bf16, fp8) : prepare_prefix(D, bf16)) !=
                      cudaSuccess)
        return BSP_ERR_CUDA;
    if (prepare_tail(D, bf16, graph ? plan->max_tail : plan->max_tail_len, Hq, fp8) != cudaSuccess) return BSP_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    PrefixParams pp{};
    if (prefix) {
        cuuint64_t qdims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(R)};
        cuuint64_t qstr[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
        // query rows per TMA box: the row block, or a quadrant's share of it (half-row softmax; the wide
        // layout's quadrants)
        const int W = plan->beam_width;
        // (a prefill on the two-block kernel: units of two blocks of beams_per_block prompt tokens)
        const int qbeams = alt    ? alt_quad_beams(D, plan->beams_per_block, G)
                           : wide ? wide_quad_beams(D, prefill ? 2 * plan->beams_per_block : W, G)
                                  : (prefill ? 0 : prefix_quad_beams(D, plan->beams_per_block, G));
        if ((alt || wide) && qbeams <= 0) return BSP_ERR_INVALID_ARG;
        cuuint32_t qbox[3] = {64, static_cast<cuuint32_t>(G),
                              static_cast<cuuint32_t>(qbeams > 0 ? qbeams : plan->beams_per_block)};
        const int ps = geo.page_size;
        // pools viewed as 2-D [pool row][head_dim]; one box = min(page, 64) rows x 64 columns (E4M3 pools:
        // x head_dim one-byte columns)
        cuuint64_t kdims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(geo.num_pages) * Hkv * ps};
        cuuint64_t kstr[1] = {static_cast<cuuint64_t>(D) * (fp8 ? 1 : 2)};
        cuuint32_t kbox[2] = {static_cast<cuuint32_t>(fp8 ? D : 64), static_cast<cuuint32_t>(std::min(ps, kTileKeys))};
        if (!encode_map(&tq, geo.dtype, 3, q, qdims, qstr, qbox) ||
            !encode_map(&tk, geo.dtype, 2, k_pool, kdims, kstr, kbox, fp8) ||
            !encode_map(&tv, geo.dtype, 2, v_pool, kdims, kstr, kbox, fp8))
            return BSP_ERR_CUDA;
        pp.k_pool = k_pool;
        pp.v_pool = v_pool;
        pp.beam_pages = beam_pages;
        pp.ci = cache_indirection;
        pp.o = o;
        pp.lse = lse;
        pp.beam_pages_stride = beam_pages_stride;
        pp.max_seq = max_seq;
        pp.lse_base2 = (flags & BSP_FLAG_LSE_BASE2) ? 1 : 0;
        pp.units = reinterpret_cast<const int32_t*>(ws + plan->off_units);
        pp.cta_off = reinterpret_cast<const int32_t*>(ws + plan->off_cta);
        pp.req = reinterpret_cast<const int32_t*>(ws + plan->off_req);
        pp.pages = reinterpret_cast<const int32_t*>(ws + plan->off_pages);
        pp.part_o = reinterpret_cast<float*>(ws + plan->off_part_o);
        pp.part_lse = reinterpret_cast<float*>(ws + plan->off_part_lse);
        pp.status = reinterpret_cast<int32_t*>(ws);
        pp.W = W;
        pp.Hq = Hq;
        pp.Hkv = Hkv;
        pp.G = G;
        pp.ps_log2 = ilog2(ps);
        pp.Wblk = wide && !prefill ? (W + 1) / 2 : plan->beams_per_block;  // beams (prompt tokens) of one MMA block
        pp.bq = qbeams;
        pp.num_pages = geo.num_pages;
        pp.num_units = graph ? 1 : plan->num_units;  // (graph: launched whatever the captured plan holds)
        if (graph) {
            pp.graph_hdr = reinterpret_cast<const int32_t*>(ws + kStatusBytes);
            pp.graph_batch = plan->batch;
        }
        pp.scale_log2 = softmax_scale * k_scale * log2e;
        pp.v_scale = v_scale;
    }
    TailParams tp{};
    tp.q = q;
    tp.k_pool = k_pool;
    tp.v_pool = v_pool;
    tp.beam_pages = beam_pages;
    tp.ci = cache_indirection;
    tp.req = reinterpret_cast<const int32_t*>(ws + plan->off_req);
    tp.part_o = reinterpret_cast<const float*>(ws + plan->off_part_o);
    tp.part_lse = reinterpret_cast<const float*>(ws + plan->off_part_lse);
    tp.o = o;
    tp.lse = lse;
    tp.status = reinterpret_cast<int32_t*>(ws);
    tp.B = plan->batch;
    tp.W = plan->beam_width;
    tp.Hq = Hq;
    tp.Hkv = Hkv;
    tp.G = G;
    tp.ps_log2 = ilog2(geo.page_size);
    tp.num_pages = geo.num_pages;
    tp.beam_pages_stride = beam_pages_stride;
    tp.max_seq = max_seq;
    tp.scale_log2 = softmax_scale * k_scale * log2e;
    tp.lse_base2 = (flags & BSP_FLAG_LSE_BASE2) ? 1 : 0;
    tp.v_scale = v_scale;
    if (graph) {
        tp.graph_hdr = reinterpret_cast<const int32_t*>(ws + kStatusBytes);
        tp.graph_max_tail = plan->max_tail;
    }

    auto record = [&](int i) -> bool { return record_event(events, i, s); };
    if (!record(0)) return BSP_ERR_CUDA;
    if (prefix) {
        const int ctas = graph ? plan->num_sms : plan->prefix_ctas;
        const cudaError_t e = alt    ? launch_alt(D, bf16, ctas, tq, tk, tv, pp, s, fp8)
                              : wide ? launch_wide(D, bf16, ctas, tq, tk, tv, pp, s, fp8)
                                   : launch_prefix(D, bf16, ctas, tq, tk, tv, pp, s);
        if (e != cudaSuccess) return BSP_ERR_CUDA;
    }
    if (!record(1)) return BSP_ERR_CUDA;
    // without timing events between them, the tail kernel overlaps the end of the prompt kernel
    if ((graph || plan->tail_requests > 0) &&
        launch_tail(D, bf16, graph ? plan->max_tail : plan->max_tail_len, tp, prefix && events == nullptr, s, fp8) !=
            cudaSuccess)
        return BSP_ERR_CUDA;
    if (!record(2)) return BSP_ERR_CUDA;
    return BSP_OK;
}
}  // namespace bsp

namespace {
// The attention of a staged plan (decode or prefill): argument checks, the launches on the plan's
// workspace, and with BSP_FLAG_CHECK the device status.
bsp_status attn_impl(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
                     int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse, void* const* events,
                     void* stream, bool prefill, bool fp8 = false, float k_scale = 1.f, float v_scale = 1.f) {
    bsp_status st = check_plan(plan);
    if (st != BSP_OK) return st;
    st = attn_check_args(plan, q, k_pool, v_pool, beam_pages, beam_pages_stride, cache_indirection, max_seq,
                         softmax_scale, flags, o, lse, prefill, fp8, k_scale, v_scale);
    if (st != BSP_OK) return st;
    if (plan->total_rows == 0) return BSP_OK;
    st = attn_launches(plan, static_cast<uint8_t*>(plan->ws_device), q, k_pool, v_pool, beam_pages, beam_pages_stride,
                       cache_indirection, max_seq, softmax_scale, flags, o, lse, events,
                       static_cast<cudaStream_t>(stream), prefill, k_scale, v_scale);
    if (st != BSP_OK) return st;
    if (flags & BSP_FLAG_CHECK) return bsp_read_device_status(plan, stream, 1, nullptr);
    return BSP_OK;
}
}  // namespace

extern "C" {

bsp_status bsp_decode_attn(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
                           int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse,
                           void* const* events, void* stream) {
    return attn_impl(plan, q, k_pool, v_pool, beam_pages, beam_pages_stride, cache_indirection, max_seq,
                     softmax_scale, flags, o, lse, events, stream, false);
}

bsp_status bsp_decode_attn_fp8(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* beam_pages, int32_t beam_pages_stride,
                               const int32_t* cache_indirection, int32_t max_seq, float softmax_scale,
                               float k_scale, float v_scale, int32_t flags, void* o, float* lse,
                               void* const* events, void* stream) {
    return attn_impl(plan, q, k_pool, v_pool, beam_pages, beam_pages_stride, cache_indirection, max_seq,
                     softmax_scale, flags, o, lse, events, stream, false, true, k_scale, v_scale);
}

bsp_status bsp_prefill_attn(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                            float softmax_scale, int32_t flags, void* o, float* lse, void* const* events,
                            void* stream) {
    return attn_impl(plan, q, k_pool, v_pool, nullptr, 0, nullptr, 0, softmax_scale, flags, o, lse, events, stream,
                     true);
}

}  // extern "C"
