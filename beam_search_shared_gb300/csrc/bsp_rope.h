// Launch contract of the RoPE append kernels (bsp_rope.cu) with the host library.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace bsp {

// RoPE on the paged append (bsp_rope.cu).
struct RopeAppendParams {
    const void* k_new;
    const void* v_new;
    int64_t src_row_stride;  // elements
    void* q;                 // may be null: no query rows
    int64_t q_row_stride;    // elements
    const int32_t* loc;
    const int32_t* pos;
    const float* cos_sin;    // [max_pos][rot]
    void* k_pool;
    void* v_pool;
    int32_t* status;
    int n, Hq, Hkv, ps_log2, num_pages;
    int rot, interleaved, max_pos;
};
cudaError_t launch_rope_append(int head_dim, bool bf16, const RopeAppendParams& p, cudaStream_t stream);
cudaError_t prepare_rope_append(int head_dim, bool bf16);
cudaError_t launch_rope_cos_sin(int max_pos, int rot, double base, float* cos_sin, cudaStream_t stream);


}  // namespace bsp
