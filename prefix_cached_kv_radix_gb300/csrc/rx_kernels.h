// Internal launch interfaces between the kernel files of libradixattn.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rx {

// Generic CUDA-core causal attention (one warp per row and head).
struct SimtParams {
    int32_t batch, hq, hkv;
    int64_t total_rows;           // extend: bound batch*max_qo_len (rows past qo_indptr[batch] exit); decode: batch
    const void* q;                // [rows, hq, D]
    const int64_t* qo_indptr;     // extend only
    const int32_t* prefix_lens;   // extend only
    const int32_t* kv_lens;       // decode only (non-null selects decode)
    const int32_t* r2t;
    int64_t stride;
    const void* k_pool;
    const void* v_pool;
    int64_t num_slots;
    void* out;
    float* lse;                   // natural log, optional
    float scale;
    int32_t max_len;              // host bound: extend max n_b, decode max L_b
    int32_t* status;
};

int launch_attn_simt(const SimtParams& p, int dtype, int head_dim, cudaStream_t stream);

}  // namespace rx
