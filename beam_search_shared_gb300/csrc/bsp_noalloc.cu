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

}  // namespace

}  // namespace bsp

extern "C" BSP_API bsp_status bsp_decode_attn_noalloc(
    const bsp_geometry* geo, int32_t batch, int32_t beam_width, const int32_t* prefix_len, const int32_t* tail_len,
    const int32_t* prefix_pages, int32_t prefix_pages_stride, int32_t max_tail, const void* q, const void* k_pool,
    const void* v_pool, const int32_t* beam_pages, int32_t beam_pages_stride, const int32_t* cache_indirection,
    int32_t max_seq, float softmax_scale, int32_t flags, void* o, float* lse, void* stream) {
    using namespace bsp;
    if (flags & ~(BSP_FLAG_LSE_BASE2 | BSP_FLAG_CHECK)) return BSP_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BSP_ERR_INVALID_ARG;
    if (geo && geo->kv_dtype != BSP_KV_DTYPE_SAME) return BSP_ERR_UNSUPPORTED;  // 16-bit pools only
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
    if (plan.total_rows == 0) return BSP_OK;
    st = attn_check_args(&plan, q, k_pool, v_pool, beam_pages, beam_pages_stride, cache_indirection, max_seq,
                         softmax_scale, flags, o, lse, false);
    if (st != BSP_OK) return st;

    uint8_t* ws = static_cast<uint8_t*>(scratch);
    // the status word must start at zero; the image and partials are rewritten before use
    if (cudaMemsetAsync(ws, 0, kStatusBytes, s) != cudaSuccess) return BSP_ERR_CUDA;
    if (cudaMemcpyAsync(ws + kStatusBytes, g_noalloc_image, plan.image_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return BSP_ERR_CUDA;
    st = attn_launches(&plan, ws, q, k_pool, v_pool, beam_pages, beam_pages_stride, cache_indirection, max_seq,
                       softmax_scale, flags, o, lse, nullptr, s, false);
    if (st != BSP_OK) return st;
    if (flags & BSP_FLAG_CHECK) {
        int32_t dflags = 0;
        if (cudaStreamSynchronize(s) != cudaSuccess) return BSP_ERR_CUDA;
        if (cudaMemcpy(&dflags, ws, sizeof dflags, cudaMemcpyDeviceToHost) != cudaSuccess) return BSP_ERR_CUDA;
        if (dflags & BSP_DEVFLAG_PAGE_INDEX) return BSP_ERR_PAGE_INDEX;
        if (dflags & BSP_DEVFLAG_TIMEOUT) return BSP_ERR_DEVICE_TIMEOUT;
    }
    return BSP_OK;
}
