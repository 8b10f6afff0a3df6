// Generic causal attention over pooled KV on CUDA cores (fp32 workloads).
//
// "Prompt Caching" (Ultralytics glossary), "How prompt caching works": each new token
// attends causally to every earlier token of its prompt, the cached prefix included; the
// cached keys/values stand in for recomputing the prefix.  Row i of request b (position
// p = P_b + i) of query head h attends keys 0..p gathered through req_to_token[b, :].
//
// One warp per (row, head); lanes split the head dimension; keys are streamed with an online
// softmax, their slots and K/V rows fetched ahead of use.  This path serves fp32 (the tiny correctness workload),
// where tensor cores would change the arithmetic; bf16 goes through the tcgen05 extend
// kernel and the mma.sync decode kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "radix_attn.h"
#include "rx_common.h"
#include "rx_device.cuh"
#include "rx_kernels.h"

namespace rx {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(128) attn_simt_kernel(SimtParams p) {
    constexpr int E = D / 32;   // elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * 4 + warp;
    if (item >= p.total_rows * p.hq) return;
    const int64_t row = item / p.hq;
    const int h = (int)(item - row * p.hq);
    const int g = h / (p.hq / p.hkv);
    int b;
    int64_t pos;
    if (p.kv_lens) {                       // decode: row b is request b's single token
        b = (int)row;
        const int32_t L = p.kv_lens[b];
        if (L < 1 || L > p.max_len || L > p.stride) {
            if (lane == 0 && h == 0) report(p.status, RX_DEV_BAD_LENGTH);
            return;
        }
        pos = L - 1;
    } else {                               // extend: find the request owning this row
        if (row >= p.qo_indptr[p.batch]) return;
        int lo = 0, hi = p.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.qo_indptr[mid] <= row) lo = mid; else hi = mid - 1;
        }
        b = lo;
        const int64_t i = row - p.qo_indptr[b];
        const int64_t n = p.qo_indptr[b + 1] - p.qo_indptr[b];
        const int64_t P = p.prefix_lens[b];
        if (n > p.max_len || P < 0 || P + n > p.stride) {
            if (lane == 0 && h == 0 && i == 0) report(p.status, RX_DEV_BAD_LENGTH);
            return;
        }
        pos = P + i;
    }
    const T* qr = (const T*)p.q + (row * p.hq + h) * D;
    float qv[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = to_f<T>(qr[lane + 32 * e]);
        acc[e] = 0.f;
    }
    const int32_t* slots = p.r2t + (int64_t)b * p.stride;
    float m = -INFINITY, l = 0.f;
    // Keys in runs of 32: one coalesced load of the run's slots (a lane each), then KG keys'
    // K and V rows requested together before the first is used, so that a key costs a
    // fraction of a memory round trip instead of two dependent ones.  The online softmax still
    // takes the keys one by one in order, with the same arithmetic as a key-at-a-time loop.
    constexpr int KG = 8;
    const int64_t nkeys = pos + 1;
    for (int64_t j0 = 0; j0 < nkeys; j0 += 32) {
        const int cnt = (int)(nkeys - j0 < 32 ? nkeys - j0 : 32);
        const int32_t s_lane = lane < cnt ? slots[j0 + lane] : 0;
        if (lane < cnt && (s_lane < 0 || s_lane >= p.num_slots)) report(p.status, RX_DEV_BAD_SLOT);
        for (int k0 = 0; k0 < cnt; k0 += KG) {
            float kv[KG][E], vv[KG][E];
            bool ok[KG];
#pragma unroll
            for (int u = 0; u < KG; ++u) {
                const int32_t s = __shfl_sync(0xffffffffu, s_lane, (k0 + u) & 31);   // the same in every lane
                ok[u] = k0 + u < cnt && s >= 0 && s < p.num_slots;
                const int64_t base = ((int64_t)(ok[u] ? s : 0) * p.hkv + g) * D;
                const T* kr = (const T*)p.k_pool + base;
                const T* vr = (const T*)p.v_pool + base;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    kv[u][e] = ok[u] ? to_f<T>(kr[lane + 32 * e]) : 0.f;
                    vv[u][e] = ok[u] ? to_f<T>(vr[lane + 32 * e]) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < KG; ++u) {
                if (!ok[u]) continue;       // a bad slot (reported) or past the row's last key
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) dot += qv[e] * kv[u][e];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                const float sc = dot * p.scale;
                const float mn = fmaxf(m, sc);
                const float corr = expf(m - mn);
                const float w = expf(sc - mn);
                l = l * corr + w;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = acc[e] * corr + w * vv[u][e];
                m = mn;
            }
        }
    }
    T* orow = (T*)p.out + (row * p.hq + h) * D;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) orow[lane + 32 * e] = from_f<T>(acc[e] * inv);
    if (p.lse && lane == 0) p.lse[row * p.hq + h] = m + logf(l);
}

int launch_attn_simt(const SimtParams& p, int dtype, int head_dim, cudaStream_t stream) {
    const int64_t items = p.total_rows * p.hq;
    if (items == 0) return RX_OK;
    const int64_t blocks = (items + 3) / 4;
    if (blocks >= (1ll << 31)) {
        set_error("attention: too many rows");
        return RX_EINVAL;
    }
    if (dtype == RX_F32 && head_dim == 64)
        attn_simt_kernel<float, 64><<<(unsigned)blocks, 128, 0, stream>>>(p);
    else if (dtype == RX_F32 && head_dim == 128)
        attn_simt_kernel<float, 128><<<(unsigned)blocks, 128, 0, stream>>>(p);
    else if (dtype == RX_BF16 && head_dim == 64)
        attn_simt_kernel<__nv_bfloat16, 64><<<(unsigned)blocks, 128, 0, stream>>>(p);
    else if (dtype == RX_BF16 && head_dim == 128)
        attn_simt_kernel<__nv_bfloat16, 128><<<(unsigned)blocks, 128, 0, stream>>>(p);
    else {
        set_error("attention: head_dim %d unsupported (64 or 128)", head_dim);
        return RX_EINVAL;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("attention: launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

}  // namespace rx
