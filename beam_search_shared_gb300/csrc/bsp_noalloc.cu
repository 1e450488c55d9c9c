// bsp_decode_attn_noalloc: the cascade decode attention for callers that must
// not allocate device memory.
//
// Some callers cannot call cudaMalloc on the decode path: serving engines that
// hand the whole GPU to their KV-cache pools at start-up and forbid later
// allocations, plugins whose host runtime owns every device allocation, and
// code that must not take the allocator's locks while it decodes. This entry
// point needs no workspace from them: its scratch (plan image, status word and
// the prompt partial states) lives in one file-scope device array of fixed
// size, and the plan image is built in a file-scope host array, so the call
// allocates nothing and calls no allocating routine.
//
// Rules that come with the shared array:
//  * the array is part of this translation unit's device module. CUDA loads
//    modules lazily by default (CUDA_MODULE_LOADING=LAZY): the driver places
//    the array on a device when the module is first used there, which is the
//    address lookup below. A caller that gives the rest of the GPU away at
//    start-up therefore makes one set-up call per device first (batch 0, any
//    valid geometry: it only looks the array up and returns), before it
//    allocates its pools. With CUDA_MODULE_LOADING=EAGER the array is placed
//    when the library's modules load. Either way the device then holds
//    kNoallocScratchBytes until the process exits;
//  * every call looks up the array's device address with the caller's device
//    current (cheap once the module is loaded), so a device reset between
//    calls leaves no stale address behind;
//  * every call uses the same array and it keeps the last call's contents:
//    the status word is cleared by each call, the rest is rewritten before it
//    is read; calls whose GPU work overlaps (other streams, other host threads)
//    race on the array, so serialise them;
//  * a call on a stream that is being captured into a CUDA graph is refused
//    (BSP_ERR_INVALID_ARG, nothing looked up or enqueued): each call copies its
//    plan from one shared host array, so a captured copy would replay whatever
//    a later call left there;
//  * device-side index errors (a bad cache_indirection value, beam page or
//    prompt page id) set the status word in the array, which only
//    BSP_FLAG_CHECK reads back (it synchronises the stream); without that flag
//    they are not reported;
//  * steps whose plan and prompt partials exceed the array are rejected with
//    BSP_ERR_CAPACITY before anything is enqueued.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/bsp.h"
#include "bsp_internal.h"

namespace bsp {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(BSP_NOALLOC_SCRATCH_MIB) << 20;
constexpr size_t kNoallocImageBytes = size_t(1) << 20;

// Device scratch shared by every call of bsp_decode_attn_noalloc on a device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// Host staging of the plan image (pageable: cudaMemcpyAsync has consumed it when it returns).
alignas(64) static uint8_t g_noalloc_image[kNoallocImageBytes];

std::mutex g_noalloc_mutex;

// Address of the device array on the current device. Looked up on every call: the first lookup on a
// device loads this file's module there (and with it the array); later ones only read the address.
bsp_status scratch_for_current_device(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return BSP_ERR_CUDA;
    }
    *out = p;
    return BSP_OK;
}

bool noalloc_device_ptr_ok(const void* p) {
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool noalloc_encode(CUtensorMap* m, int dtype, int rank, const void* base, const cuuint64_t* dims,
                    const cuuint64_t* strides, const cuuint32_t* box) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    if (!enc) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dtype == BSP_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
               static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int noalloc_log2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

}  // namespace

// bsp_host.cpp: a decode plan with the packed layout (no fixed offsets for graph replays)
bsp_status plan_build_packed(const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len,
                             const int32_t* tail_len, const int32_t* prefix_pages, int32_t prefix_pages_stride,
                             int32_t max_tail, int32_t num_sms, void* image, size_t image_bytes, bsp_plan_t* out);
}  // namespace bsp

extern "C" BSP_API bsp_status bsp_decode_attn_noalloc(
    const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len, const int32_t* tail_len,
    const int32_t* prefix_pages, int32_t prefix_pages_stride, int32_t max_tail, const void* q, const void* k_pool,
    const void* v_pool, const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
    int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse, void* stream) {
    using namespace bsp;
    if (flags & ~(BSP_FLAG_LSE_BASE2 | BSP_FLAG_CHECK)) return BSP_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BSP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        // a captured call would record a copy from the shared host plan array: refused
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        const cudaError_t e = cudaStreamIsCapturing(s, &cs);
        if (e == cudaErrorStreamCaptureImplicit) {
            cudaGetLastError();
            return BSP_ERR_INVALID_ARG;  // the legacy stream while another stream captures
        }
        if (e != cudaSuccess) {
            cudaGetLastError();
            return BSP_ERR_CUDA;
        }
        if (cs != cudaStreamCaptureStatusNone) return BSP_ERR_INVALID_ARG;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    void* scratch = nullptr;
    bsp_status st = scratch_for_current_device(&scratch);
    if (st != BSP_OK) return st;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BSP_ERR_CUDA;

    bsp_plan_t plan;
    // the packed layout: this entry point is never replayed from a graph, and the scratch is fixed
    st = bsp::plan_build_packed(geo, batch, beam_width, prefix_len, tail_len, prefix_pages, prefix_pages_stride, max_tail,
                           sms, g_noalloc_image, kNoallocImageBytes, &plan);
    if (st != BSP_OK) return st;
    if (plan.device_bytes_used > kNoallocScratchBytes) return BSP_ERR_CAPACITY;
    const int64_t R = static_cast<int64_t>(batch) * beam_width;
    if (R == 0) return BSP_OK;
    if (!noalloc_device_ptr_ok(q) || !noalloc_device_ptr_ok(k_pool) || !noalloc_device_ptr_ok(v_pool) ||
        !noalloc_device_ptr_ok(o) || !noalloc_device_ptr_ok(lse))
        return BSP_ERR_INVALID_ARG;
    if (plan.max_tail_len > 0) {
        if (!noalloc_device_ptr_ok(beam_pages) || !noalloc_device_ptr_ok(cache_indirection)) return BSP_ERR_INVALID_ARG;
        if (max_seq < plan.max_total_len || max_seq < 1) return BSP_ERR_INVALID_ARG;
        if (beam_pages_stride < (plan.max_total_len + geo->page_size - 1) / geo->page_size) return BSP_ERR_INVALID_ARG;
    }

    uint8_t* ws = static_cast<uint8_t*>(scratch);
    // the status word must start at zero; the image and partials are rewritten before use
    if (cudaMemsetAsync(ws, 0, kStatusBytes, s) != cudaSuccess) return BSP_ERR_CUDA;
    if (cudaMemcpyAsync(ws + kStatusBytes, g_noalloc_image, plan.image_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return BSP_ERR_CUDA;

    const int D = geo->head_dim, Hq = geo->num_q_heads, Hkv = geo->num_kv_heads, G = Hq / Hkv;
    const bool bf16 = geo->dtype == BSP_DTYPE_BF16;
    const float log2e = 1.4426950408889634f;
    const int ps = geo->page_size;
    if (plan.num_units > 0) {
        CUtensorMap tq, tk, tv;
        cuuint64_t qdims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(R)};
        cuuint64_t qstr[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
        // query rows per TMA box: the row block, or a quadrant's share of it (half-row softmax)
        const int qbeams = prefix_quad_beams(D, plan.beams_per_block, G);
        cuuint32_t qbox[3] = {64, static_cast<cuuint32_t>(G),
                              static_cast<cuuint32_t>(qbeams > 0 ? qbeams : plan.beams_per_block)};
        cuuint64_t kdims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(geo->num_pages) * Hkv * ps};
        cuuint64_t kstr[1] = {static_cast<cuuint64_t>(D) * 2};
        cuuint32_t kbox[2] = {64, static_cast<cuuint32_t>(ps < kTileKeys ? ps : kTileKeys)};
        if (!noalloc_encode(&tq, geo->dtype, 3, q, qdims, qstr, qbox) ||
            !noalloc_encode(&tk, geo->dtype, 2, k_pool, kdims, kstr, kbox) ||
            !noalloc_encode(&tv, geo->dtype, 2, v_pool, kdims, kstr, kbox))
            return BSP_ERR_CUDA;
        PrefixParams pp{};
        pp.k_pool = k_pool;
        pp.v_pool = v_pool;
        pp.beam_pages = beam_pages;
        pp.ci = cache_indirection;
        pp.o = o;
        pp.lse = lse;
        pp.beam_pages_stride = beam_pages_stride;
        pp.max_seq = max_seq;
        pp.lse_base2 = (flags & BSP_FLAG_LSE_BASE2) ? 1 : 0;
        pp.units = reinterpret_cast<const int32_t*>(ws + plan.off_units);
        pp.cta_off = reinterpret_cast<const int32_t*>(ws + plan.off_cta);
        pp.req = reinterpret_cast<const int32_t*>(ws + plan.off_req);
        pp.pages = reinterpret_cast<const int32_t*>(ws + plan.off_pages);
        pp.part_o = reinterpret_cast<float*>(ws + plan.off_part_o);
        pp.part_lse = reinterpret_cast<float*>(ws + plan.off_part_lse);
        pp.status = reinterpret_cast<int32_t*>(ws);
        pp.W = beam_width;
        pp.Hq = Hq;
        pp.Hkv = Hkv;
        pp.G = G;
        pp.ps_log2 = noalloc_log2(ps);
        pp.Wblk = plan.beams_per_block;
        pp.bq = qbeams;
        pp.num_pages = geo->num_pages;
        pp.num_units = plan.num_units;
        pp.scale_log2 = softmax_scale * log2e;
        if (prepare_prefix(D, bf16) != cudaSuccess ||
            launch_prefix(D, bf16, plan.prefix_ctas, tq, tk, tv, pp, s) != cudaSuccess)
            return BSP_ERR_CUDA;
    }
    TailParams tp{};
    tp.q = q;
    tp.k_pool = k_pool;
    tp.v_pool = v_pool;
    tp.beam_pages = beam_pages;
    tp.ci = cache_indirection;
    tp.req = reinterpret_cast<const int32_t*>(ws + plan.off_req);
    tp.part_o = reinterpret_cast<const float*>(ws + plan.off_part_o);
    tp.part_lse = reinterpret_cast<const float*>(ws + plan.off_part_lse);
    tp.o = o;
    tp.lse = lse;
    tp.status = reinterpret_cast<int32_t*>(ws);
    tp.B = batch;
    tp.W = beam_width;
    tp.Hq = Hq;
    tp.Hkv = Hkv;
    tp.G = G;
    tp.ps_log2 = noalloc_log2(ps);
    tp.num_pages = geo->num_pages;
    tp.beam_pages_stride = beam_pages_stride;
    tp.max_seq = max_seq;
    tp.scale_log2 = softmax_scale * log2e;
    tp.lse_base2 = (flags & BSP_FLAG_LSE_BASE2) ? 1 : 0;
    if (plan.tail_requests > 0 && (prepare_tail(D, bf16, plan.max_tail_len, Hq) != cudaSuccess ||
                                   launch_tail(D, bf16, plan.max_tail_len, tp, plan.num_units > 0, s) != cudaSuccess))
        return BSP_ERR_CUDA;
    if (flags & BSP_FLAG_CHECK) {
        int32_t dflags = 0;
        if (cudaStreamSynchronize(s) != cudaSuccess) return BSP_ERR_CUDA;
        if (cudaMemcpy(&dflags, ws, sizeof dflags, cudaMemcpyDeviceToHost) != cudaSuccess) return BSP_ERR_CUDA;
        if (dflags & BSP_DEVFLAG_PAGE_INDEX) return BSP_ERR_PAGE_INDEX;
        if (dflags & BSP_DEVFLAG_TIMEOUT) return BSP_ERR_DEVICE_TIMEOUT;
    }
    return BSP_OK;
}
