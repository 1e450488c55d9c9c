/*
 * bsp.h - C ABI of the GB300 shared-prefix (cascade) beam decode attention
 * library (libbsp.so).
 *
 * One decode step of wide beam search over a paged KV cache, per layer:
 *   bsp_plan        host planning: validates lengths and beam 0's prompt page
 *                   tables, splits the prompt attention into work units and
 *                   stages the plan to the device without a stream sync;
 *   bsp_append_kv   writes each beam's new token K/V at its flat cache slot;
 *   bsp_decode_attn attends each request's shared prompt once for all of its
 *                   beams (tensor cores), each beam's own tail through
 *                   cache_indirection, and merges the two by log-sum-exp,
 *                   returning O and LSE.
 * The method: TensorRT-LLM PR #21738, "Add opt-in cascade attention for wide
 * beam search on KVCM V2" (description, "Solution"); the valid-prefix bound:
 * TensorRT-Model-Connect PR #2202, "prefill and decode over the cached prefix,
 * not the whole KV allocation"; the append: TensorRT-LLM PR #18614, "Fuse
 * MiniMax-M3 MSA per-layer KV-cache writes into one kernel".
 *
 * Conventions for every call
 *  - Memory: all device and host memory is owned by the caller. The library
 *    allocates nothing and keeps no state between calls beyond what it writes
 *    into the caller's workspace.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Every device effect of a call is enqueued on that stream; no call
 *    synchronises the stream unless documented (BSP_FLAG_CHECK,
 *    bsp_read_device_status).
 *  - Errors: arguments are validated on the host before anything is enqueued;
 *    on any error nothing is launched and pools/outputs are left unchanged.
 *    Indices that live in device memory (beam_pages, cache_indirection,
 *    out_cache_loc) cannot be validated without a sync: kernels bounds-check
 *    them, skip the access and set a flag in the workspace's device status
 *    word, which bsp_read_device_status (or BSP_FLAG_CHECK) reports as
 *    BSP_ERR_PAGE_INDEX. Kernels never trap.
 *  - Layouts (row-major, innermost last, 16-bit elements unless stated):
 *      q, o            [R = batch * beam_width][num_q_heads][head_dim], row r = b*W + w
 *      lse             [R][num_q_heads] float32
 *      k_pool, v_pool  [num_pages][num_kv_heads][page_size][head_dim]
 *      beam_pages      [R][beam_pages_stride] int32 page ids of each beam's sequence
 *      cache_indirection [batch][beam_width][max_seq] int32 source beam per position
 *    Query head h uses kv head h / (num_q_heads / num_kv_heads).
 *    Device pointers must be 16-byte aligned.
 */
#ifndef BSP_H_
#define BSP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BSP_API __attribute__((visibility("default")))
#else
#define BSP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bsp_status {
    BSP_OK = 0,
    BSP_ERR_INVALID_ARG = 1,  /* null/misaligned/host pointer, bad length or stride */
    BSP_ERR_UNSUPPORTED = 2,  /* dtype, head_dim, group size, page size or tail outside the supported set */
    BSP_ERR_PAGE_INDEX = 3,   /* a page id, slot, indirection value or RoPE position out of range */
    BSP_ERR_CAPACITY = 4,     /* workspace or staging buffer too small */
    BSP_ERR_STALE_PLAN = 5,   /* plan superseded by a newer bsp_plan on the same workspace */
    BSP_ERR_CUDA = 6,         /* a CUDA runtime/driver call failed */
    BSP_ERR_DEVICE_TIMEOUT = 7 /* a kernel's bounded wait gave up (reported by status reads) */
} bsp_status;

enum { BSP_DTYPE_BF16 = 0, BSP_DTYPE_FP16 = 1 };
/* What the K/V pools hold (bsp_geometry.kv_dtype): elements of `dtype`, or one-byte FP8 E4M3 values
   ("e4m3fn": 4 exponent bits with bias 7, 3 fraction bits, no infinities, max 448) in the same
   [page][kv head][slot][head_dim] layout */
enum { BSP_KV_DTYPE_SAME = 0, BSP_KV_DTYPE_E4M3 = 1 };

/* bsp_decode_attn flags */
enum {
    BSP_FLAG_LSE_BASE2 = 1, /* write LSE as log2-sum-exp2 instead of the natural log */
    BSP_FLAG_CHECK = 2,     /* synchronise after the launches and report device status */
    BSP_FLAG_GRAPH = 4      /* bsp_decode_attn only, not with BSP_FLAG_CHECK: launch shapes that do not
                               depend on the plan's lengths, so that the launches may be captured in a
                               CUDA graph once and replayed after every later bsp_plan on the same
                               workspace with the same batch, beam_width, max_tail, geometry, SM count,
                               page-table stride and buffers (the CUDA-graph serving mode: TensorRT-LLM
                               PR #21738, description: the host plan of a step is made before capture and
                               before every replay; the tail bound caps the tail under graphs). The
                               prompt kernel runs one CTA per SM of the plan and the tail kernel is
                               always launched for max_tail tail rows; a replay whose staged plan has
                               another shape writes nothing and sets BSP_DEVFLAG_GRAPH */
};

#define BSP_MAX_TAIL 8   /* tail positions per beam (TensorRT-LLM PR #21738, description: correctness and limits) */
#define BSP_MAX_GROUP 8  /* query heads per kv head */

/* Bits of the device status word. */
#define BSP_DEVFLAG_PAGE_INDEX 1
#define BSP_DEVFLAG_TIMEOUT 2
#define BSP_DEVFLAG_POSITION 4  /* a RoPE position outside [0, max_position) (bsp_rope_append_kv) */
#define BSP_DEVFLAG_GRAPH 8     /* a replayed graph-mode launch found a plan of another shape (nothing
                                   written); reported as BSP_ERR_STALE_PLAN */

typedef struct bsp_geometry {
    int32_t num_q_heads;  /* Hq */
    int32_t num_kv_heads; /* Hkv; Hq % Hkv == 0, Hq / Hkv <= BSP_MAX_GROUP */
    int32_t head_dim;     /* 64, 128 or 256 */
    int32_t page_size;    /* tokens per page: 8, 16, 32, 64 or 128 */
    int32_t num_pages;    /* pages in each pool */
    int32_t dtype;        /* BSP_DTYPE_*; q, o and new K/V share it, and the pools unless kv_dtype says */
    int32_t kv_dtype;     /* BSP_KV_DTYPE_*: 0 (the pools hold `dtype`), or E4M3 pools, which decode
                             plans at head_dim 64 and 128 support (bsp_decode_attn_fp8; the writes:
                             bsp_append_kv_fp8, bsp_rope_append_kv_fp8); any other use returns
                             BSP_ERR_UNSUPPORTED */
} bsp_geometry;

/*
 * Plan of one decode step, filled by bsp_plan / bsp_plan_build. Caller-owned
 * plain data; the fields below `generation` describe the staged device image
 * and are read by the launches. A plan refers to the workspace it was staged
 * into; it stays valid until the next bsp_plan on that workspace.
 */
typedef struct bsp_plan_t {
    bsp_geometry geo;
    int32_t batch;               /* B */
    int32_t beam_width;          /* W (a prefill plan: the rows of a partial slot, the largest prompt) */
    int32_t max_tail;            /* bound on every tail_len, <= BSP_MAX_TAIL */
    int32_t prefix_pages_stride; /* row stride of the prefix_pages table given to the plan */
    int32_t num_units;           /* prompt-attention work units (CTAs) */
    int32_t num_parts;           /* (request, key split) prompt partial states */
    int32_t row_blocks;          /* query-row blocks per (request, kv head) */
    int32_t beams_per_block;     /* beams in one query-row block */
    int32_t tile_keys;           /* keys per prompt tile */
    int32_t max_prefix_len;      /* max_b P_b */
    int32_t max_total_len;       /* max_b P_b + T_b */
    int32_t num_sms;             /* SM count the units were balanced for */
    int32_t max_tail_len;        /* max_b T_b */
    int32_t prefix_ctas;         /* persistent CTAs of the prompt kernel (<= num_sms) */
    uint64_t generation;         /* staging generation of this plan (0: built only, not staged) */
    void* ws_device;             /* device workspace the plan was staged into */
    uint64_t ws_device_bytes;
    void* ws_host;               /* host staging buffer paired with ws_device */
    uint64_t image_bytes;        /* bytes of the staged plan image */
    uint64_t off_req;            /* byte offsets into ws_device */
    uint64_t off_units;
    uint64_t off_pages;
    uint64_t off_part_lse;
    uint64_t off_part_o;
    uint64_t device_bytes_used;
    int32_t tail_requests;       /* requests the tail kernel finishes (no prompt, a prompt split over
                                    several partial states, or more tail keys per row block than one
                                    tile holds); the prompt kernel finishes the others. No tail launch
                                    when 0 */
    int32_t total_rows;          /* query rows of the step: batch * beam_width (decode) or the prompt
                                    tokens of all requests (prefill) */
    int32_t kind;                /* 0: a decode-step plan (bsp_plan); 1: a prefill plan (bsp_plan_prefill) */
    int32_t layout;              /* prompt kernel of the plan: 0 one softmax warp set (head_dim 256, and
                                    decode row blocks of <= 64 query rows, two threads per row); 2 two
                                    MMA blocks in one CTA sharing every K/V tile: all 129-256 query rows
                                    of a (request, kv head) of a decode step (the prompt read once), or
                                    a prefill's prompt tokens at head_dim <= 128 in units of two blocks
                                    of beams_per_block = 4 * floor(32 / G) tokens; 1 two softmax warp
                                    sets taking a unit's key tiles alternately (other decode steps at
                                    head_dim <= 128) */
    uint64_t off_cta;            /* byte offset of the per-CTA unit table */
    uint64_t reserved;
} bsp_plan_t;

/* Human-readable name of a bsp_status value. Never NULL. */
BSP_API const char* bsp_status_string(int32_t status);

/*
 * Rows to bind for a cached prefix of `valid_rows` rows in an allocation of
 * `capacity` rows: the next multiple of 256 rows, or a single row when nothing
 * is cached, at most the allocation (TensorRT-Model-Connect PR #2202,
 * Implementation: kv_cache.{h,cpp}, kCacheRowBucket). The kernels themselves
 * read only the valid rows; this is the bound a caller binds when it needs a
 * shape that changes once per 256 tokens. Returns -1 if capacity < 1.
 */
BSP_API int32_t bsp_bucket_rows(int32_t valid_rows, int32_t capacity);

/*
 * Upper bounds of the device workspace and the host staging buffer for plans
 * with batch <= max_batch, beam_width <= max_beam and prompt page tables of at
 * most max_prefix_pages pages (TensorRT-LLM PR #21738: the fp32 workspace is
 * sized once from the engine's largest row counts). The host staging buffer should
 * be pinned (page-locked) for the copy to be asynchronous.
 */
BSP_API bsp_status bsp_workspace_size(const bsp_geometry* geo, int32_t max_batch, int32_t max_beam,
                              int32_t max_prefix_pages, size_t* device_bytes, size_t* host_bytes);

/*
 * Host-only planning: validates the step and writes the device plan image into
 * `image` (host memory, `image_bytes` capacity) without touching CUDA. Used by
 * bsp_plan; exposed for tests and for callers that stage the image themselves.
 *   prefix_len[b]   valid prompt rows P_b >= 0 of request b (host)
 *   tail_len[b]     tail positions T_b in [0, max_tail] (host); the tail
 *                   includes the current token once it is appended
 *   prefix_pages    host [batch][prefix_pages_stride]: beam 0's page ids of the
 *                   prompt; the first ceil(P_b / page_size) entries of row b
 *                   are read and each must lie in [0, num_pages), else
 *                   BSP_ERR_PAGE_INDEX (never clamped) (TensorRT-LLM PR #21738,
 *                   the commit that makes an invalid prompt page id an error)
 *   max_tail        <= BSP_MAX_TAIL (the same PR's limit on the generated
 *                   positions a beam may hold in graph mode)
 *   num_sms         SMs to balance the prompt work units for (> 0)
 * `plan_out->generation` is 0 and the workspace fields are left NULL.
 */
BSP_API bsp_status bsp_plan_build(const bsp_geometry* geo, int32_t batch, int32_t beam_width,
                          const int32_t* prefix_len, const int32_t* tail_len, const int32_t* prefix_pages,
                          int32_t prefix_pages_stride, int32_t max_tail, int32_t num_sms, void* image,
                          size_t image_bytes, bsp_plan_t* plan_out);

/*
 * Plans one decode step (per-step host planning, TensorRT-LLM PR #21738: the
 * plan is made on the host before graph capture and before each replay, and its
 * inputs are staged in pinned memory so that planning every step never
 * synchronises the stream).
 * Builds the image (bsp_plan_build, balanced for the current device's SM
 * count), writes it into one of two slots of `ws_host` and enqueues its copy
 * into `ws_device` on `stream`. The workspace pair (ws_device, ws_host) must
 * have at least the sizes bsp_workspace_size reports; ws_host should be pinned.
 * A slot is rewritten only after the stream has finished copying the plan
 * that used it two plans earlier (the stream echoes a generation number back
 * into ws_host); if that has not happened the call waits for it, up to 10 s,
 * then returns BSP_ERR_CUDA. Planning again makes every earlier plan of this
 * workspace stale (BSP_ERR_STALE_PLAN from the launches) (TensorRT-LLM PR
 * #21738, the commit that discards the previous step's plan).
 */
BSP_API bsp_status bsp_plan(const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len,
                    const int32_t* tail_len, const int32_t* prefix_pages, int32_t prefix_pages_stride,
                    int32_t max_tail, void* ws_device, size_t ws_device_bytes, void* ws_host,
                    size_t ws_host_bytes, void* stream, bsp_plan_t* plan_out);

/*
 * Per-step update of a staged decode plan: the same batch, beam width, prompt
 * lengths and prompt pages, new tail lengths. Beam search keeps a request's
 * prompt fixed while its tail grows by one position a step, so the work units,
 * the CTA table and the prompt page list of the plan (the dealing, which costs
 * the planner O(units log units) and more) stay as they are; only the request
 * records change: T_b, and whether the prompt kernel or the tail kernel
 * finishes request b (the same rule bsp_plan applies). O(batch) host work and
 * one copy of the image header and request records (64 + 48 * batch bytes)
 * through the next staging slot, with the slot protocol of bsp_plan (TensorRT-
 * LLM PR #21738: per-step host planning with pinned staging and no stream
 * synchronisation). The units stay balanced for the tails the plan was built
 * with; re-plan with bsp_plan when the batch or a prompt changes.
 *   plan       in/out: a current decode plan of its workspace (from bsp_plan or
 *              an earlier update); on success its generation, max_tail_len,
 *              max_total_len and tail_requests describe the new step and
 *              every earlier plan of the workspace is stale
 *   tail_len   host [batch]: T_b in [0, plan->max_tail] (BSP_ERR_CAPACITY
 *              above it, BSP_ERR_INVALID_ARG below 0); nothing is changed on
 *              error
 *   stream     the stream of the step's launches (the copy is enqueued on it)
 * A CUDA graph captured with BSP_FLAG_GRAPH from a plan of this workspace
 * replays correctly after updates: the header it checks does not change.
 */
BSP_API bsp_status bsp_plan_update_tails(bsp_plan_t* plan, const int32_t* tail_len, void* stream);

/*
 * Paged KV append: for every new token i < n and kv head h, copies the
 * head_dim elements of k_new / v_new row i, head h to
 * pool[out_cache_loc[i] / page_size][h][out_cache_loc[i] % page_size][:],
 * bit for bit, in one launch (TensorRT-LLM PR #18614, description: one launch
 * per layer computes each slot's page and in-page row from out_cache_loc in
 * registers and writes K and V in the same pass).
 *   k_new, v_new    device [n] rows of num_kv_heads * head_dim contiguous
 *                   elements, rows `src_row_stride` elements apart
 *                   (>= num_kv_heads * head_dim, a multiple of 8), so that K
 *                   and V may be column slices of one projection output
 *   out_cache_loc   device int32 [n] flat slots; a slot outside
 *                   [0, num_pages * page_size) is skipped and flagged
 *   n               0 is a no-op returning BSP_OK; must be <= batch * beam_width
 *   events          NULL, or 2 cudaEvent_t (as void*) recorded on `stream`
 *                   before and after the append kernel (timing only; under
 *                   stream capture they become external event-record nodes)
 * Duplicate slots are a caller error (the surviving row is unspecified).
 */
BSP_API bsp_status bsp_append_kv(const bsp_plan_t* plan, const void* k_new, const void* v_new, int64_t src_row_stride,
                         const int32_t* out_cache_loc, int32_t n, void* k_pool, void* v_pool,
                         void* const* events, void* stream);

/*
 * Paged append into FP8 E4M3 pools (a KV cache kept in 8 bits; TensorRT-LLM
 * PR #18614, the review follow-up commit on the fused KV write: the
 * case of an fp8 source written to an fp8 cache, and the review of msa_scatter.py: the
 * write converts the source dtype to the cache's). Same slots, layout and
 * error behaviour as bsp_append_kv, with pools of one byte per element,
 * uint8 [num_pages][num_kv_heads][page_size][head_dim]:
 *   src_dtype = BSP_FP8_SRC_16BIT: k_new / v_new hold the geometry's dtype
 *                   (bf16 or fp16); element x is stored as the E4M3 value
 *                   nearest to fp32(x) * k_mul (v_mul for V), the product
 *                   rounded once to fp32, ties to even, values past +-448
 *                   saturated to +-448 (k_mul, v_mul finite and > 0: a cache's
 *                   per-tensor quantisation multipliers, 1 for a plain cast)
 *   src_dtype = BSP_FP8_SRC_E4M3: k_new / v_new hold E4M3 bytes, copied bit
 *                   for bit (the multipliers are not used)
 *   src_row_stride  elements of the source type between rows, >= num_kv_heads
 *                   * head_dim, rows 16-byte aligned (a multiple of 8 for a
 *                   16-bit source, of 16 for E4M3)
 * The plan may have either kv_dtype (the pools passed here are E4M3 either way);
 * bsp_decode_attn_fp8 reads such pools.
 */
enum { BSP_FP8_SRC_16BIT = 0, BSP_FP8_SRC_E4M3 = 1 };
BSP_API bsp_status bsp_append_kv_fp8(const bsp_plan_t* plan, const void* k_new, const void* v_new,
                                     int64_t src_row_stride, int32_t src_dtype, float k_mul, float v_mul,
                                     const int32_t* out_cache_loc, int32_t n, void* k_pool, void* v_pool,
                                     void* const* events, void* stream);

/*
 * Rotary position embedding (RoPE) on the paged append. The pages apply RoPE to
 * K before it is written to the paged cache (TensorRT-LLM PR #21738: the model
 * applies it itself, per the description; the review of flash_attn4_kernels.py
 * names the rope_write_kv_paged helper and its partial-RoPE partner lookup) but
 * do not define it; the definition is the published one (Su et al., RoFormer,
 * section 3.2): the first rotary_dim dims of a head row form rotary_dim/2 pairs,
 * pair j turns by the angle p * theta_j, theta_j = base^(-2j / rotary_dim),
 * (x, y) -> (x cos - y sin, y cos + x sin); the other dims pass unchanged.
 *
 * The caller-owned table of cos/sin values, device fp32
 *   cos_sin[p][j]                  = cos(p * theta_j),  j < rotary_dim / 2
 *   cos_sin[p][rotary_dim / 2 + j] = sin(p * theta_j),
 * p in [0, max_position), is filled once by bsp_rope_cos_sin.
 */
typedef struct bsp_rope_config {
    const float* cos_sin;   /* device [max_position][rotary_dim], 16-byte aligned */
    int32_t max_position;   /* rows of cos_sin */
    int32_t rotary_dim;     /* rotated leading dims of a head row: a multiple of 16, 16 .. head_dim */
    int32_t interleaved;    /* 0: pair j = dims (j, j + rotary_dim/2) (rotate-half, e.g. Qwen3);
                               1: pair j = dims (2j, 2j + 1) */
    int32_t reserved;       /* 0 */
} bsp_rope_config;

/*
 * Fills the cos/sin table of a bsp_rope_config: angles and their cos/sin in
 * fp64 on the device, each value rounded once to fp32. One launch on `stream`,
 * no sync.
 *   max_position   > 0 rows;  rotary_dim even, 2 .. 1024;  base > 1, finite
 *   cos_sin        device fp32 [max_position][rotary_dim], 16-byte aligned
 * Argument errors: BSP_ERR_INVALID_ARG before any launch.
 */
BSP_API bsp_status bsp_rope_cos_sin(int32_t max_position, int32_t rotary_dim, double base, float* cos_sin,
                                    void* stream);

/*
 * Paged append with RoPE, one launch: for every new token i < n at position
 * positions[i] and slot out_cache_loc[i], the kv head rows of k_new are rotated
 * and written, the rows of v_new copied, to
 * pool[slot / page_size][h][slot % page_size][:] (as bsp_append_kv); when q is
 * non-NULL, the token's num_q_heads query rows are rotated in place. Rotation
 * in fp32 from the fp32 table (one fused multiply-add per output after one
 * product), rounded to nearest even into the pools' dtype; V rows and dims past
 * rotary_dim are copied bit for bit.
 *   plan            a decode or prefill plan (geometry, status word, n bound)
 *   rope            table and layout (bsp_rope_config)
 *   positions       device int32 [n]: the token's logical position (a decode
 *                   step: P_b + T_b - 1 for every beam of request b; a
 *                   prefill: C_b + t)
 *   q               NULL, or device [n] rows of num_q_heads * head_dim elements
 *                   q_row_stride elements apart (>= that, a multiple of 8)
 *   k_new, v_new, src_row_stride, out_cache_loc, n, k_pool, v_pool, events:
 *                   as bsp_append_kv
 * A token whose slot is outside [0, num_pages * page_size) or whose position is
 * outside [0, max_position) is skipped entirely (no pool row written, its q rows
 * left as they were) and sets BSP_DEVFLAG_PAGE_INDEX or BSP_DEVFLAG_POSITION;
 * bsp_read_device_status reports either as BSP_ERR_PAGE_INDEX. Host-checkable
 * errors return before any launch with nothing written.
 */
BSP_API bsp_status bsp_rope_append_kv(const bsp_plan_t* plan, const bsp_rope_config* rope, const int32_t* positions,
                                      void* q, int64_t q_row_stride, const void* k_new, const void* v_new,
                                      int64_t src_row_stride, const int32_t* out_cache_loc, int32_t n,
                                      void* k_pool, void* v_pool, void* const* events, void* stream);

/*
 * RoPE on the append into FP8 E4M3 pools (the fused write of the FP8 KV path:
 * TensorRT-LLM PR #18614, the review follow-up commit on the fused KV
 * write, where the RoPE kernel writes K and V as E4M3). As bsp_rope_append_kv, except that
 * k_pool / v_pool are uint8 E4M3 pools: each rotated K value (fp32, not rounded
 * to 16 bits first) times k_mul and each V value times v_mul, the product
 * rounded to fp32, is stored as the nearest E4M3 value (ties to even,
 * saturating at +-448); q (if given) is rotated in place in its 16-bit dtype.
 * k_mul, v_mul finite and > 0. Errors as bsp_rope_append_kv.
 */
BSP_API bsp_status bsp_rope_append_kv_fp8(const bsp_plan_t* plan, const bsp_rope_config* rope, const int32_t* positions,
                                          void* q, int64_t q_row_stride, const void* k_new, const void* v_new,
                                          int64_t src_row_stride, float k_mul, float v_mul,
                                          const int32_t* out_cache_loc, int32_t n, void* k_pool, void* v_pool,
                                          void* const* events, void* stream);

/*
 * Cascade decode attention (TensorRT-LLM PR #21738, description, "Solution"):
 * for every row r = b*W + w and query head h,
 *   O[r][h] = softmax(scale * q K^T) V over the beam's logical sequence:
 *             prompt positions j < P_b read through beam 0's prompt pages
 *             (the plan's prefix_pages), tail positions j in [P_b, P_b + T_b)
 *             read through beam_pages[b*W + cache_indirection[b][w][j]];
 *   LSE[r][h] = log-sum-exp of the scaled scores (natural log, or base 2 with
 *             BSP_FLAG_LSE_BASE2); an empty sequence gives O = 0, LSE = -inf.
 * Each (request, kv head) reads its prompt keys a single time for all beams and query
 * heads (tensor cores), the tail per beam, and the two merge exactly by
 * log-sum-exp. Only the valid P_b prompt rows are read, never the allocation.
 *   beam_pages_stride  entries per beam_pages row, >= ceil(max(P_b+T_b)/page_size)
 *   max_seq            innermost extent of cache_indirection, >= max(P_b + T_b)
 *   softmax_scale      > 0, typically 1/sqrt(head_dim)
 *   flags              BSP_FLAG_* bits
 *   events             NULL, or 3 cudaEvent_t (as void*) recorded on `stream`
 *                      before the prompt kernel, between the prompt and the
 *                      tail kernels, and after the tail kernel (timing only;
 *                      under stream capture they become external event-record
 *                      nodes)
 * The plan must be the latest one staged into its workspace.
 */
BSP_API bsp_status bsp_decode_attn(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
                           int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse,
                           void* const* events, void* stream);

/*
 * bsp_decode_attn over FP8 E4M3 pools (TensorRT-LLM PR #18614, the review
 * follow-up commit on the fused KV write: a KV cache kept in 8 bits, written by
 * bsp_append_kv_fp8). The plan's geometry has kv_dtype = BSP_KV_DTYPE_E4M3 (and
 * head_dim 64 or 128); k_pool and v_pool hold one byte per element. Key and
 * value element x of the pools stand for e4m3(x) * k_scale and
 * e4m3(x) * v_scale (per-tensor scales, finite and > 0; 1 and 1 read the codes
 * as they are). The result is the decode attention of bsp_decode_attn over
 * those keys and values:
 *   O   = softmax(softmax_scale * k_scale * q . e4m3(K)) e4m3(V) * v_scale
 *   LSE = log-sum-exp of softmax_scale * k_scale * q . e4m3(K)
 * The kernels read the E4M3 tiles (half the bytes of the 16-bit pools) and
 * widen them exactly to the q dtype in shared memory (every E4M3 value is a
 * bf16 and a binary16 value), so the tensor-core products are those of the
 * 16-bit path. A NaN code (0x7f, 0xff) in a key or value row that is read
 * makes that row's output NaN. Other arguments, flags, events and errors as
 * bsp_decode_attn; a plan whose pools are not E4M3 is BSP_ERR_INVALID_ARG here,
 * and an E4M3 plan is BSP_ERR_INVALID_ARG for bsp_decode_attn, bsp_append_kv
 * and bsp_rope_append_kv.
 */
BSP_API bsp_status bsp_decode_attn_fp8(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* beam_pages, int32_t beam_pages_stride,
                               const int32_t* cache_indirection, int32_t max_seq, float softmax_scale,
                               float k_scale, float v_scale, int32_t flags, void* o, float* lse,
                               void* const* events, void* stream);

/*
 * Prefill over the cached prefix (TensorRT-Model-Connect PR #2202, "prefill and
 * decode over the cached prefix, not the whole KV allocation", Implementation:
 * the prompt rows attend the bound cache rows and then the prompt rows, with
 * only the valid cached prefix bound). Request b holds cached_len[b] >= 0 valid
 * cached rows and prompt_len[b] >= 0 prompt tokens, whose K/V the caller has
 * already written (bsp_append_kv) at logical positions cached_len[b] ..
 * cached_len[b] + prompt_len[b] - 1; every position p of request b is read
 * through its page table: page = pages[b * pages_stride + p / page_size],
 * slot = p % page_size (the first ceil((cached + prompt) / page_size) entries
 * must lie in [0, num_pages), else BSP_ERR_PAGE_INDEX). With `causal` != 0,
 * prompt token i sees positions 0 .. cached_len[b] + i, else all
 * cached_len[b] + prompt_len[b] positions. Positions past those are never
 * read. The query rows are the prompt tokens of all requests in order (request
 * b's tokens start at the sum of the earlier prompt_len), `total_rows` in all.
 * A request whose longest work unit is above the launch's mean load per SM has
 * its cached rows cut into key ranges (every cut inside the cached rows, so
 * that each prompt row has keys in each range); the prompt kernel writes one
 * partial state per range and the tail kernel merges them (the plan's
 * tail_requests counts such requests, its beam_width is then the rows of a
 * partial slot: the largest prompt_len). bsp_plan_prefill_build writes the host
 * image only (as bsp_plan_build); bsp_plan_prefill stages it without a sync (as
 * bsp_plan); the workspace must hold a plan of max_batch = batch and max_beam =
 * 1 (bsp_workspace_size), and with max_beam = the largest prompt_len it also
 * holds the partial states of key splits: bsp_plan_prefill plans without them
 * when they do not fit.
 */
BSP_API bsp_status bsp_plan_prefill_build(const bsp_geometry* geo, int32_t batch, const int32_t* cached_len,
                                  const int32_t* prompt_len, const int32_t* pages, int32_t pages_stride,
                                  int32_t causal, int32_t num_sms, void* image, size_t image_bytes,
                                  bsp_plan_t* plan_out);
BSP_API bsp_status bsp_plan_prefill(const bsp_geometry* geo, int32_t batch, const int32_t* cached_len,
                            const int32_t* prompt_len, const int32_t* pages, int32_t pages_stride,
                            int32_t causal, void* ws_device, size_t ws_device_bytes, void* ws_host,
                            size_t ws_host_bytes, void* stream, bsp_plan_t* plan_out);

/*
 * The prefill attention of a bsp_plan_prefill plan: for every prompt row r and
 * query head h, O[r][h] = softmax(scale * q K^T) V and LSE[r][h] over the keys
 * the plan gives that row, on the tensor cores (the prompt kernel: at head_dim
 * <= 128 each (request, kv head, two blocks of 4 * floor(32 / G) prompt tokens,
 * key range) a work unit of the two-block kernel, at 256 each (request, kv
 * head, block of floor(128 / G) tokens, key range) one of the one-set kernel; a
 * causal unit reads keys only up to its last token; then the tail kernel for
 * the requests whose keys were split). q, o [total_rows][Hq][head_dim]
 * in the pools' dtype, lse [total_rows][Hq] fp32 (natural log, or base 2 with
 * BSP_FLAG_LSE_BASE2). A decode plan is BSP_ERR_INVALID_ARG here (and a prefill
 * plan in bsp_decode_attn). events: NULL or 3 cudaEvent_t, as bsp_decode_attn.
 */
BSP_API bsp_status bsp_prefill_attn(const bsp_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
                            float softmax_scale, int32_t flags, void* o, float* lse, void* const* events,
                            void* stream);

/*
 * Synchronises `stream`, then reads the workspace's device status word into
 * *flags_out (BSP_DEVFLAG_* bits set by kernels since the last clear) and
 * clears it when `clear` is non-zero. Returns BSP_ERR_PAGE_INDEX or
 * BSP_ERR_DEVICE_TIMEOUT when a bit is set, BSP_OK otherwise.
 */
BSP_API bsp_status bsp_read_device_status(const bsp_plan_t* plan, void* stream, int32_t clear, int32_t* flags_out);

/* Size, in MiB, of the fixed device scratch array of bsp_decode_attn_noalloc (one per GPU). */
#define BSP_NOALLOC_SCRATCH_MIB 32

/*
 * bsp_decode_attn_noalloc - the same cascade decode attention as
 * bsp_decode_attn, for callers that cannot allocate device memory.
 * (This entry point has no counterpart on the pages the method comes from.)
 *
 * Some callers cannot call cudaMalloc on the decode path: serving engines that
 * give the whole GPU to their KV-cache pools at start-up and forbid later
 * allocations, plugins whose host runtime owns every device allocation, and
 * code that must not take the allocator's locks while it decodes. This call
 * takes no workspace: it plans the step itself (the arguments of bsp_plan) and
 * keeps its scratch (plan image, status word, prompt partial states) in one
 * fixed device array of BSP_NOALLOC_SCRATCH_MIB MiB compiled into the library.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Set-up: CUDA loads a library's device code lazily by default
 *    (CUDA_MODULE_LOADING=LAZY), and the array is placed on a device when this
 *    call first looks it up there. So call it once per device with batch = 0
 *    (and a valid geometry; nothing else is read) before allocating the KV
 *    pools: that call only looks the array up, with the device current, and
 *    returns BSP_OK. (With CUDA_MODULE_LOADING=EAGER the array is placed when
 *    the library is loaded.) From then on the device holds the array until the
 *    process exits. Every call looks the address up again, so no address
 *    outlives a device reset.
 *  - All calls share the array, which keeps the last call's contents; the call
 *    clears the status word itself. Calls whose GPU work overlaps (different
 *    streams or host threads) race on the array: serialise them.
 *  - A call on a stream that is being captured into a CUDA graph returns
 *    BSP_ERR_INVALID_ARG before anything is looked up or enqueued: each call
 *    copies its plan from one shared host array, so a captured copy would
 *    replay a later call's plan.
 *  - Indices in device memory (cache_indirection, beam_pages) are checked by
 *    the kernels as in bsp_decode_attn, and a bad one sets a bit in the array's
 *    status word; only BSP_FLAG_CHECK (which synchronises the stream) reads it
 *    back, as BSP_ERR_PAGE_INDEX. Without that flag such errors go unreported.
 *  - A step whose plan image and prompt partials need more than the array is
 *    rejected with BSP_ERR_CAPACITY before anything is enqueued.
 * Inputs, outputs, layouts, flags (BSP_FLAG_LSE_BASE2, BSP_FLAG_CHECK) and
 * errors are otherwise those of bsp_plan and bsp_decode_attn; the plan arrays
 * are host memory, every other pointer device memory. The plan image is copied
 * from host memory that is not page-locked. 16-bit pools only: a geometry with
 * E4M3 pools is BSP_ERR_UNSUPPORTED here.
 */
BSP_API bsp_status bsp_decode_attn_noalloc(const bsp_geometry* geo, int32_t batch, int32_t beam_width,
                                           const int32_t* prefix_len, const int32_t* tail_len,
                                           const int32_t* prefix_pages, int32_t prefix_pages_stride,
                                           int32_t max_tail, const void* q, const void* k_pool,
                                           const void* v_pool, const int32_t* beam_pages, int32_t beam_pages_stride,
                                           const int32_t* cache_indirection, int32_t max_seq, float softmax_scale,
                                           int32_t flags, void* o, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSP_H_ */
