// Internal launch interfaces between the kernel files of libradixattn.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "radix_attn.h"

namespace rx {

// Set-up that a CUDA context keeps per device (a kernel's dynamic shared-memory limit and
// carve-out, a device capability check): done once on each device, under a lock, so that a
// process driving several GPUs from several threads sets it on every device it launches on.
// Devices 0..63; a later context on the same device (after cudaDeviceReset) is not tracked.
struct PerDeviceOnce {
    std::mutex mu;
    uint64_t done = 0;        // bit d: set-up succeeded on device d
};

// Runs f() (returning an RX_* status) the first time it is called with device `dev` current;
// later calls on that device return RX_OK without running it.  A failed f() is retried on the
// next call.
template <class F>
int per_device_once(PerDeviceOnce& o, F&& f) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return f();
    std::lock_guard<std::mutex> lk(o.mu);
    if (o.done & (1ull << dev)) return RX_OK;
    const int rc = f();
    if (rc == RX_OK) o.done |= 1ull << dev;
    return rc;
}

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

// Shared-prefix part on the tcgen05 kernel: for every group, its query rows (stacked) attend
// one chunk of the group's shared keys (slot-table row grp_src[g]); fp32 normalised partials
// and log2-domain lse go to part_o/part_lse at partial index part_base + chunk.
struct SharedTcParams {
    const void* q;                // [batch, hq, D] bf16
    const int32_t* r2t;
    int64_t stride;
    const void* k_pool;
    const void* v_pool;
    int64_t num_slots;
    int32_t batch, hq, hkv, head_dim;
    float scale;
    int32_t* status;
    int32_t num_groups, max_group_rows;
    const int32_t* grp_row_indptr;   // [num_groups+1] into grp_rows
    const int32_t* grp_rows;         // global query-row ids (decode: request ids)
    const int32_t* grp_src;          // [num_groups] slot-table row holding the shared slots
    const int32_t* grp_len;
    int32_t chunk, n_chunks;
    float* part_o;
    float* part_lse;
    int32_t part_per, part_base;
};

int launch_shared_prefix_tc(const SharedTcParams& p, cudaStream_t stream);

// Small extend (decode_attention.cu): every request's new tokens times the query heads of a kv
// head fit 8 rows and its keys one 1024-key chunk (guaranteed by r2t_stride <= 1024).
constexpr int SMALL_EXT_MAX_ROWS = 8;
constexpr int SMALL_EXT_MAX_KEYS = 1024;
struct SmallExtendArgs {
    const void* q;
    const int64_t* qo_indptr;
    const int32_t* prefix_lens;
    const int32_t* r2t;
    int64_t stride;
    const void* k_pool;
    const void* v_pool;
    int64_t num_slots;
    void* out;
    float* lse;
    int32_t batch, hq, hkv, head_dim, max_qo_len;
    float scale;
    int32_t* status;
};
int launch_extend_small(const SmallExtendArgs& a, cudaStream_t stream);


// kv_pool_write for the requests of one call whose new tokens are t_begin .. t_end-1 (index
// arrays absolute: a slice of a step's requests passes its offset pointers).  With stage_bytes
// > 0 the same launch also copies stage_src (16-byte aligned, any device-readable address, e.g.
// the device mapping of a pinned staging buffer) to stage_dst; the index arrays it reads itself
// must then not be inside stage_dst.
int kv_pool_write_rows(const rx_attn_desc* desc, int32_t batch, const int32_t* d_prefix_slots,
                       const int64_t* d_prefix_indptr, const int32_t* d_new_slots, const int64_t* d_qo_indptr,
                       const void* d_k_new, const void* d_v_new, void* d_k_pool, void* d_v_pool, int32_t* d_req_to_token,
                       int64_t r2t_stride, int64_t t_begin, int64_t t_end, int32_t* d_status, cudaStream_t stream,
                       const void* stage_src = nullptr, void* stage_dst = nullptr, int64_t stage_bytes = 0,
                       unsigned* done_ctr = nullptr, uint32_t* done_flag = nullptr, uint32_t done_seq = 0);

}  // namespace rx
