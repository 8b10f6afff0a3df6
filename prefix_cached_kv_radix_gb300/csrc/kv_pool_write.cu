// kv_pool_write: per-request slot table plus scatter of the new tokens' K/V into the pools.
//
// "Prompt Caching" (Ultralytics glossary), "How prompt caching works": only the new
// tokens' keys/values are computed; the cached prefix is reused.  Here the new rows are
// written once into their pool slots, and each request's slot table lists its matched
// (shared) slots followed by its new slots, so attention can gather the whole context.
//
// One launch, three kinds of blocks: optionally, a few blocks first copy a step's staging
// buffer (its index arrays, read through the device mapping of pinned host memory) to its
// device copy for the kernels that follow -- the step runtime's small device-row steps, where
// the table blocks read the slot lists from the mapped buffer themselves -- then batch * tiles
// blocks each fill one tile of
// KPW_TILE entries of a table row (coalesced int32 stores; each thread has KPW_PER
// independent loads in flight, so a long row is not one block's chain of dependent round
// trips); the rest copy 16-byte vectors of the new K/V rows to their slots (consecutive
// threads copy consecutive vectors of a row: coalesced reads, and full 32-byte sectors on
// the scattered writes).  HBM-bound: the algorithmic bytes are 2 * T * hkv * head_dim * elt
// read + the same written + the table.  When the index arrays are read from a pinned staging
// buffer, the launch can end by writing a sequence number to pinned host memory once every
// block is done with them, so that the host reuses the buffer without a CUDA event.
#include <cuda_runtime.h>

#include <algorithm>

#include "radix_attn.h"
#include "rx_common.h"
#include "rx_device.cuh"
#include "rx_kernels.h"

namespace rx {

constexpr int KPW_THREADS = 256;
constexpr int KPW_TILE = KPW_THREADS * 4;            // table entries per block (4 per thread)

// One tile of NT * 4 entries of request b's slot-table row: its matched (prefix) slots, then
// its new slots, then -1 up to the row's stride.  All loads are issued before the first store
// (each thread has 4 independent loads in flight).  Bad lengths and slots are reported; a bad
// entry is written as -1.
template <int NT>
__device__ __forceinline__ void kpw_table_tile(int b, int64_t tile, const int32_t* __restrict__ prefix_slots,
                                               const int64_t* __restrict__ prefix_indptr,
                                               const int32_t* __restrict__ new_slots,
                                               const int64_t* __restrict__ qo_indptr, int32_t* __restrict__ r2t,
                                               int64_t stride, int64_t num_slots, int64_t t_begin, int64_t t_end,
                                               int32_t* status) {
    constexpr int PER = 4;
    const int64_t j0 = tile * NT * PER;
    const int64_t p0 = prefix_indptr[b], P = prefix_indptr[b + 1] - p0;
    const int64_t q0 = qo_indptr[b], n = qo_indptr[b + 1] - q0;
    int32_t* row = r2t + (int64_t)b * stride;
    const bool bad_len = P < 0 || n < 0 || P + n > stride || q0 < t_begin || q0 + n > t_end;
    if (bad_len && j0 == 0 && threadIdx.x == 0) report(status, RX_DEV_BAD_LENGTH);
    int32_t s[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {          // the loads first, all in flight together
        const int64_t j = j0 + threadIdx.x + (int64_t)u * NT;
        s[u] = -1;
        if (!bad_len && j < P)
            s[u] = prefix_slots[p0 + j];
        else if (!bad_len && j < P + n)
            s[u] = new_slots[q0 + (j - P)];
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int64_t j = j0 + threadIdx.x + (int64_t)u * NT;
        if (j >= stride) break;
        if (s[u] < -1 || s[u] >= num_slots || (s[u] == -1 && !bad_len && j < P + n)) {
            report(status, RX_DEV_BAD_SLOT);
            s[u] = -1;
        }
        row[j] = s[u];
    }
}

// The new tokens' K/V rows t_begin .. t_end-1 (the rows of this call's requests) to their
// slots: copy block `cb` of `ncb`.  Consecutive threads copy consecutive 16-byte vectors of a
// row (coalesced reads, full 32-byte sectors on the scattered writes).
__device__ __forceinline__ void kv_copy_rows(int64_t cb, int64_t ncb, const int32_t* __restrict__ new_slots,
                                             const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                             uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int64_t num_slots,
                                             int32_t row_vecs, int64_t t_begin, int64_t t_end, int32_t* status) {
    const int64_t nvec = (t_end - t_begin) * row_vecs;
    const int64_t step = ncb * blockDim.x;
    for (int64_t j = cb * blockDim.x + threadIdx.x; j < nvec; j += step) {
        const int64_t i = t_begin * row_vecs + j;
        const int64_t t = i / row_vecs;
        const int32_t v = (int32_t)(i - t * row_vecs);
        const int32_t s = new_slots[t];
        if (s < 0 || s >= num_slots) {
            if (v == 0) report(status, RX_DEV_BAD_SLOT);
            continue;
        }
        const int64_t dst = (int64_t)s * row_vecs + v;
        k_pool[dst] = k_new[i];
        v_pool[dst] = v_new[i];
    }
}

// End of a block that read a pinned staging buffer's index arrays (every value it loaded from
// them has been consumed): the last block of the launch to get here writes `seq` to pinned
// host memory, telling the host the launch no longer reads them -- the host may then write the
// next step's arrays into the same buffer without a CUDA event.  The counter is reset for the
// buffer's next launch, which the host makes only after it has seen the flag.  Every thread of
// the block calls it.
__device__ __forceinline__ void signal_stage_done(unsigned* done_ctr, uint32_t* done_flag, uint32_t done_seq) {
    if (!done_ctr) return;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(done_ctr, 1u) == gridDim.x - 1) {
            atomicExch(done_ctr, 0u);
            __threadfence_system();
            *(volatile uint32_t*)done_flag = done_seq;
        }
    }
}

__global__ void __launch_bounds__(KPW_THREADS) kv_pool_write_kernel(
    int32_t batch, int32_t tiles, const int32_t* __restrict__ prefix_slots, const int64_t* __restrict__ prefix_indptr,
    const int32_t* __restrict__ new_slots, const int64_t* __restrict__ qo_indptr, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
    int32_t* __restrict__ r2t, int64_t stride, int64_t num_slots, int32_t row_vecs, int64_t t_begin, int64_t t_end,
    int32_t* status, const uint4* __restrict__ stage_src, uint4* __restrict__ stage_dst, int64_t stage_vecs,
    int32_t stage_blocks, unsigned* done_ctr, uint32_t* done_flag, uint32_t done_seq) {
    // a kernel launched after this one with programmatic serialization (the small-extend
    // attention) may start its own set-up now; it waits for this grid before it reads the
    // table or the pools
    pdl_launch_dependents();
    const int32_t bid = (int32_t)blockIdx.x - stage_blocks;
    const int64_t table_blocks = (int64_t)batch * tiles;
    if ((int32_t)blockIdx.x < stage_blocks) {          // the staging buffer to its device copy
        const int64_t step = (int64_t)stage_blocks * blockDim.x;
        int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        for (; i + 3 * step < stage_vecs; i += 4 * step) {   // four loads in flight per thread
            const uint4 a = stage_src[i], b = stage_src[i + step], c = stage_src[i + 2 * step], d = stage_src[i + 3 * step];
            stage_dst[i] = a;
            stage_dst[i + step] = b;
            stage_dst[i + 2 * step] = c;
            stage_dst[i + 3 * step] = d;
        }
        for (; i < stage_vecs; i += step) stage_dst[i] = stage_src[i];
    } else if ((int64_t)bid < table_blocks) {
        kpw_table_tile<KPW_THREADS>((int)(bid / tiles), bid % tiles, prefix_slots, prefix_indptr, new_slots, qo_indptr,
                                    r2t, stride, num_slots, t_begin, t_end, status);
    } else {
        kv_copy_rows(bid - table_blocks, gridDim.x - stage_blocks - table_blocks, new_slots, k_new, v_new, k_pool,
                     v_pool, num_slots, row_vecs, t_begin, t_end, status);
    }
    signal_stage_done(done_ctr, done_flag, done_seq);
}

}  // namespace rx

namespace rx {

int kv_pool_write_rows(const rx_attn_desc* desc, int32_t batch, const int32_t* d_prefix_slots,
                       const int64_t* d_prefix_indptr, const int32_t* d_new_slots, const int64_t* d_qo_indptr,
                       const void* d_k_new, const void* d_v_new, void* d_k_pool, void* d_v_pool, int32_t* d_req_to_token,
                       int64_t r2t_stride, int64_t t_begin, int64_t t_end, int32_t* d_status, cudaStream_t stream,
                       const void* stage_src, void* stage_dst, int64_t stage_bytes, unsigned* done_ctr,
                       uint32_t* done_flag, uint32_t done_seq) {
    RX_REQUIRE(desc && batch >= 0 && r2t_stride >= 0 && t_begin >= 0 && t_end >= t_begin, "kv_pool_write: bad arguments");
    RX_REQUIRE(desc->dtype == RX_F32 || desc->dtype == RX_BF16, "kv_pool_write: unknown dtype %d", desc->dtype);
    RX_REQUIRE(desc->hkv > 0 && desc->head_dim > 0 && desc->num_slots > 0, "kv_pool_write: bad shape");
    const int64_t row_bytes = (int64_t)desc->hkv * desc->head_dim * (desc->dtype == RX_F32 ? 4 : 2);
    RX_REQUIRE(row_bytes % 16 == 0, "kv_pool_write: K/V row of %lld bytes is not a multiple of 16",
               (long long)row_bytes);
    if (batch == 0) return RX_OK;
    RX_REQUIRE(d_prefix_indptr && d_qo_indptr && d_req_to_token, "kv_pool_write: null device pointer");
    RX_REQUIRE(t_end == t_begin || (d_new_slots && d_k_new && d_v_new && d_k_pool && d_v_pool),
               "kv_pool_write: null device pointer");
    for (const void* p : {d_k_new, d_v_new, (const void*)d_k_pool, (const void*)d_v_pool})
        RX_REQUIRE(((uintptr_t)p & 15) == 0, "kv_pool_write: K/V buffers must be 16-byte aligned");
    const int32_t row_vecs = (int32_t)(row_bytes / 16);
    const int64_t nvec = (t_end - t_begin) * row_vecs;
    int64_t copy_blocks = (nvec + KPW_THREADS - 1) / KPW_THREADS;
    if (copy_blocks > 152 * 16) copy_blocks = 152 * 16;
    if (copy_blocks < 1) copy_blocks = 1;
    const int64_t tiles = std::max<int64_t>(1, (r2t_stride + KPW_TILE - 1) / KPW_TILE);
    RX_REQUIRE(stage_bytes == 0 || (stage_src && stage_dst && stage_bytes % 16 == 0 && ((uintptr_t)stage_src & 15) == 0 &&
                                    ((uintptr_t)stage_dst & 15) == 0),
               "kv_pool_write: staging copy must be 16-byte aligned whole vectors");
    const int64_t stage_vecs = stage_bytes / 16;
    const int32_t stage_blocks =
        stage_vecs > 0 ? (int32_t)std::min<int64_t>(64, (stage_vecs + KPW_THREADS * 4 - 1) / (KPW_THREADS * 4)) : 0;
    const int64_t grid = stage_blocks + (int64_t)batch * tiles + copy_blocks;
    RX_REQUIRE(grid < (1ll << 31) && tiles < (1ll << 31), "kv_pool_write: batch or stride too large");
    kv_pool_write_kernel<<<(unsigned)grid, KPW_THREADS, 0, stream>>>(
        batch, (int32_t)tiles, d_prefix_slots, d_prefix_indptr, d_new_slots, d_qo_indptr, (const uint4*)d_k_new,
        (const uint4*)d_v_new, (uint4*)d_k_pool, (uint4*)d_v_pool, d_req_to_token, r2t_stride, desc->num_slots,
        row_vecs, t_begin, t_end, d_status, (const uint4*)stage_src, (uint4*)stage_dst, stage_vecs, stage_blocks,
        done_flag ? done_ctr : nullptr, done_flag, done_seq);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("kv_pool_write: launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

}  // namespace rx

extern "C" int kv_pool_write(const rx_attn_desc* desc, int32_t batch, const int32_t* d_prefix_slots,
                             const int64_t* d_prefix_indptr, const int32_t* d_new_slots,
                             const int64_t* d_qo_indptr, const void* d_k_new, const void* d_v_new, void* d_k_pool,
                             void* d_v_pool, int32_t* d_req_to_token, int64_t r2t_stride, int64_t total_new,
                             int32_t* d_status, void* stream) {
    RX_TRACE("kv_pool_write");
    RX_REQUIRE(total_new >= 0, "kv_pool_write: bad arguments");
    return rx::kv_pool_write_rows(desc, batch, d_prefix_slots, d_prefix_indptr, d_new_slots, d_qo_indptr, d_k_new,
                                  d_v_new, d_k_pool, d_v_pool, d_req_to_token, r2t_stride, 0, total_new, d_status,
                                  (cudaStream_t)stream);
}
