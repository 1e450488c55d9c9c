// Launch contract of the write-side kernels beside the plain append (RoPE on the append in
// bsp_rope.cu, the append into FP8 E4M3 pools in bsp_append.cu) with the host library.
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
    float k_mul, v_mul;      // fp8 pools: quantisation multipliers of K (after the rotation) and V
};
// fp8: the pools are E4M3 bytes (K and V quantised), else the q dtype
cudaError_t launch_rope_append(int head_dim, bool bf16, bool fp8, const RopeAppendParams& p, cudaStream_t stream);
cudaError_t prepare_rope_append(int head_dim, bool bf16, bool fp8);
cudaError_t launch_rope_cos_sin(int max_pos, int rot, double base, float* cos_sin, cudaStream_t stream);

// Append into E4M3 pools (bsp_append.cu).
struct AppendFp8Params {
    const void* k_new;       // 16-bit (bf16 / fp16) or E4M3 rows
    const void* v_new;
    int64_t src_row_stride;  // elements of the source type
    const int32_t* loc;
    uint8_t* k_pool;         // [num_pages][Hkv][ps][D] bytes
    uint8_t* v_pool;
    int32_t* status;
    float k_mul, v_mul;      // quantisation multipliers of a 16-bit source
    int n, Hkv, D, ps_log2, num_pages;
};
// src: 0 bf16, 1 fp16, 2 E4M3 (copied)
cudaError_t launch_append_fp8(int src, const AppendFp8Params& p, cudaStream_t stream);
cudaError_t prepare_append_fp8(int src);


}  // namespace bsp
