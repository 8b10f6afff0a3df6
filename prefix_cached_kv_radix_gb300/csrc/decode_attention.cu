// Split-KV decode attention over the pooled KV cache, on mma.sync tensor-core tiles.
//
// "Prompt Caching" (Ultralytics glossary), "How prompt caching works": in decode each new
// token attends to all keys and values cached for its prompt.  With RadixAttention the
// cached prefix rows live once in the pool and requests gather them through their slot
// tables ("SGLang: Efficient Execution of Structured Language Model Programs", RadixAttention).
//
// Design (GB300): the step is HBM-bound (each K/V byte is used by the hq/hkv query heads of
// one kv head only), so the kernel is built around streaming: one CTA per (request, kv head,
// chunk of keys); 16-byte cp.async gathers of 64-key stages into a 2-stage 128B-swizzled
// ring, three CTAs per SM; each warp owns 16 keys of a stage and computes S^T = K Q^T with keys in the M
// dimension of m16n8k16 (the <= 8 query heads of the group fill N, so only half of each
// tile is padding), then O^T += V^T P^T with V^T fragments from ldmatrix.trans and P^T
// moved into B-fragment layout by movmatrix.  Online softmax in the exp2 domain.  Each CTA
// writes its chunk's normalised output and log-sum-exp; a second kernel merges the chunks:
//   M = max_s lse_s, w_s = 2^(lse_s - M), o = sum_s w_s o_s / sum_s w_s.
// Groups of requests sharing a cached prefix (rx_shared_groups) get their shared run
// processed once per group on the tcgen05 kernel (extend_attention.cu, shared-prefix mode):
// the members' query rows are stacked into dense 128-row tiles, so each shared K/V row is
// read once per 256 stacked rows instead of once per request; the merge kernel adds that
// partial to each member's private chunks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "radix_attn.h"
#include "rx_common.h"
#include "rx_device.cuh"
#include "rx_kernels.h"

namespace rx {

constexpr int DEC_THREADS = 128;   // 4 warps
constexpr int DEC_STAGE_KEYS = 64; // 16 keys per warp per stage
// cp.async ring depth.  Two 32 KB stages per CTA keep the shared memory at ~69 KB, so three
// CTAs share an SM (192 KB in flight) and cover one another's prologue (length, group and slot
// loads) and epilogue (cross-warp merge): with three stages and two CTAs per SM those phases
// left the SM half idle for ~22 % of each CTA's life.
constexpr int DEC_NS = 2;
constexpr int DEC_MAX_CHUNK = SMALL_EXT_MAX_KEYS;   // keys per split (the slot list is staged in smem)
constexpr float LOG2E = 1.4426950408889634f;

__host__ __device__ constexpr int dec_ring_bytes(int D) {
    // K/V ring, or the cross-warp merge buffer that reuses it, whichever is larger
    // (the merge buffer: partial rows of D + 4 floats, running max and sum, merge weights, row lse)
    return (DEC_NS * 2 * DEC_STAGE_KEYS * D * 2) > (4 * 8 * (D + 4) * 4 + 4 * 8 * 2 * 4 + 4 * 8 * 4 + 8 * 4)
               ? (DEC_NS * 2 * DEC_STAGE_KEYS * D * 2)
               : (4 * 8 * (D + 4) * 4 + 4 * 8 * 2 * 4 + 4 * 8 * 4 + 8 * 4);
}
constexpr float LN2 = 0.6931471805599453f;

struct DecodeParams {
    const __nv_bfloat16* q;     // [batch, hq, D]
    const int32_t* r2t;
    int64_t stride;
    const int32_t* kv_lens;
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    int64_t num_slots;
    int32_t batch, hq, hkv, group;
    float scale_log2;
    int32_t chunk;              // keys per split (multiple of DEC_STAGE_KEYS)
    int32_t max_chunks;         // private partial slots per (request, head)
    int32_t max_len;
    float* part_o;              // [batch, hq, max_chunks + group_chunks, D]
    float* part_lse;            // [batch, hq, max_chunks + group_chunks] (log2 domain)
    int32_t* status;
    // shared-prefix groups
    int32_t num_groups;
    const int32_t* grp_indptr;
    const int32_t* grp_members;
    const int32_t* grp_len;
    int32_t grp_chunks;         // shared partial slots per (request, head)
    int32_t grp_rows_max;       // max stacked rows (members * group) of a group
    const int32_t* shared_of;   // [batch] keys each request takes from its group's shared run
                                // (0 outside groups; workspace, filled by the group-map kernel)
    int32_t* group_src;         // [num_groups] first member (its slot-table row holds the shared slots)
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)(chunk ^ (row & 7)); }

// Gather one stage of K and V (64 keys starting at chunk-relative key k0) into smem.
// Slot ids come from the chunk's slot list staged in shared memory (slot_s): reading them
// from global memory here would put one dependent round trip before every copy.  The list
// is checked when it is staged and padded with -1 (no key: past the chunk's end, or a bad
// slot, already reported) to the end of the last stage, so that no copy repeats the check:
// a -1 slot copies zeros.  col = g * D + this thread's 16-byte column * 8, the same for
// every key.
template <int D>
__device__ __forceinline__ void dec_load_stage(const DecodeParams& p, const int32_t* slot_s, int k0, int64_t col,
                                               uint32_t kbuf, uint32_t vbuf, int tid) {
    constexpr int CPR = D / 8;                       // 16-byte chunks per row
    constexpr int PER = DEC_STAGE_KEYS * CPR / DEC_THREADS;
    const int c = tid % CPR;
    const int64_t row_elems = (int64_t)p.hkv * D;
#pragma unroll
    for (int x = 0; x < PER; ++x) {
        const int key = tid / CPR + x * (DEC_THREADS / CPR);
        const int32_t s = slot_s[k0 + key];
        const int64_t off = (int64_t)max(s, 0) * row_elems + col;
        const uint32_t so = (uint32_t)(key * D * 2) + swz(key, c) * 16;
        const uint32_t bytes = s >= 0 ? 16u : 0u;
        cp_async_16(kbuf + so, p.k_pool + off, bytes);
        cp_async_16(vbuf + so, p.v_pool + off, bytes);
    }
}

// A slot from a slot-table row, checked against the pool: out of range, it is reported and
// becomes -1 (its key reads as zeros).
__device__ __forceinline__ int32_t checked_slot(const DecodeParams& p, int32_t s) {
    if (s < 0 || s >= p.num_slots) {
        report(p.status, RX_DEV_BAD_SLOT);
        return -1;
    }
    return s;
}

// Where the rows of a tile live (row indices into [rows, D] arrays).  Decode: row n is query
// head g*group + n of request b (head0 = b*hq + g*group), and its partial goes to slot
// (head0 + n)*per + chunk.  Small extend: row n is new token n / group, head g*group +
// n % group (head0 = g*group) of a request whose first new token is qo0, and its final
// output row is its query row.
struct DecRowMap {
    int64_t head0, per, chunk;
    __device__ __forceinline__ int64_t q_row(int n) const { return head0 + n; }
    __device__ __forceinline__ int64_t out_row(int n) const { return (head0 + n) * per + chunk; }
};
struct ExtRowMap {
    int64_t qo0;
    int hq, head0, group;
    __device__ __forceinline__ int64_t q_row(int n) const { return (qo0 + n / group) * hq + head0 + n % group; }
    __device__ __forceinline__ int64_t out_row(int n) const { return q_row(n); }
};

// Causal limits of the rows of a small extend tile: row n may see keys <= pos0 + n / group.
struct ExtRows {
    int pos0, group;
    __nv_bfloat16* out;   // final output rows ([T * hq, D])
    float* lse;           // optional natural-log lse per output row
    bool pair_store;      // out is 4-byte aligned: two bf16 per store
};

// Attention of up to 8 query rows (packed into N of m16n8k16) over keys [k_begin, k_end)
// of one slot-table row.  Decode (EXT = false): rows are the query heads of one kv head of
// one request, all keys visible; writes normalised partial outputs and log2-domain lse at
// partial slot rows.out_row(n).  Small extend (EXT = true): rows are (new token, head) pairs
// of one request with causal limits (ExtRows), the chunk covers every key, and the final
// bf16 output row rows.out_row(n) (and its lse) is written directly.
template <int D, bool EXT = false, class RowMap>
__device__ __forceinline__ void dec_chunk(const DecodeParams& p, const int32_t* slots_row, int k_begin, int k_end,
                                          int g, const RowMap& rows, int nrows, unsigned char* smem, int32_t* slot_s,
                                          ExtRows ext = ExtRows{}, bool slots_staged = false) {
    constexpr int KSTEPS = D / 16;
    constexpr int MT = D / 16;                        // m-tiles of O^T
    constexpr int ROWB = D * 2;
    constexpr int STAGE_B = DEC_STAGE_KEYS * ROWB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t4 = lane & 3, r8 = lane >> 2;
    const uint32_t sbase = smem_u32(smem);
    auto kbuf = [&](int st) { return sbase + (uint32_t)(st * 2 * STAGE_B); };
    auto vbuf = [&](int st) { return sbase + (uint32_t)(st * 2 * STAGE_B + STAGE_B); };

    // Q^T fragments (B operand of S^T = K Q^T): row n = r8, dims 16s + 2*t4 (+1), (+8).
    uint32_t qb[KSTEPS][2];
    {
        const bool valid = r8 < nrows;
        const __nv_bfloat16* qr = p.q + (valid ? rows.q_row(r8) * D : 0);
#pragma unroll
        for (int s = 0; s < KSTEPS; ++s) {
            qb[s][0] = valid ? *reinterpret_cast<const uint32_t*>(qr + 16 * s + 2 * t4) : 0u;
            qb[s][1] = valid ? *reinterpret_cast<const uint32_t*>(qr + 16 * s + 8 + 2 * t4) : 0u;
        }
    }
    float o[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows 2*t4, 2*t4+1

    const int nk = k_end - k_begin;                  // <= DEC_MAX_CHUNK
    const int nstages = (nk + DEC_STAGE_KEYS - 1) / DEC_STAGE_KEYS;
    if (!slots_staged)
        for (int i = tid; i < nstages * DEC_STAGE_KEYS; i += DEC_THREADS)
            slot_s[i] = i < nk ? checked_slot(p, slots_row[k_begin + i]) : -1;
    // the last key each of this lane's two rows may see, plus one: the chunk's end, and
    // extending, the row's own position
    int end0 = k_end, end1 = k_end;
    if (EXT) {
        end0 = min(k_end, ext.pos0 + (2 * t4) / ext.group + 1);
        end1 = min(k_end, ext.pos0 + (2 * t4 + 1) / ext.group + 1);
    }
    const int64_t col = (int64_t)g * D + (tid % (D / 8)) * 8;
    __syncthreads();
#pragma unroll
    for (int s = 0; s < DEC_NS - 1; ++s) {
        if (s < nstages) dec_load_stage<D>(p, slot_s, s * DEC_STAGE_KEYS, col, kbuf(s), vbuf(s), tid);
        cp_async_commit();
    }
    for (int it = 0; it < nstages; ++it) {
        // Every warp is done with stage it-1, whose buffer takes stage it+DEC_NS-1; issuing it
        // before waiting for stage it keeps all DEC_NS stages in flight.
        __syncthreads();
        {
            const int nx = it + DEC_NS - 1;
            if (nx < nstages)
                dec_load_stage<D>(p, slot_s, nx * DEC_STAGE_KEYS, col, kbuf(nx % DEC_NS), vbuf(nx % DEC_NS), tid);
            cp_async_commit();
        }
        cp_async_wait<DEC_NS - 1>();   // stage it has landed (this thread's copies) ...
        __syncthreads();               // ... and every thread's
        const int st = it % DEC_NS;
        const int key0 = k_begin + it * DEC_STAGE_KEYS + warp * 16;   // first key of this warp
        if (key0 >= k_end) continue;                                   // nothing for this warp
        // S^T (16 keys x 8 rows)
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int mi = lane >> 3, rr = lane & 7;
            const int krow = warp * 16 + (mi & 1) * 8 + rr;
#pragma unroll
            for (int s = 0; s < KSTEPS; ++s) {
                uint32_t a[4];
                const int ch = 2 * s + (mi >> 1);
                ldmatrix_x4(kbuf(st) + (uint32_t)(krow * ROWB) + swz(krow, ch) * 16, a[0], a[1], a[2], a[3]);
                mma_bf16_16816(sacc, a, qb[s][0], qb[s][1]);
            }
        }
        // scale, mask keys past each row's limit, online softmax per query row (column)
        const int kl = key0 + r8, kh = key0 + r8 + 8;
        float x0 = kl < end0 ? sacc[0] * p.scale_log2 : -INFINITY;
        float x1 = kl < end1 ? sacc[1] * p.scale_log2 : -INFINITY;
        float x2 = kh < end0 ? sacc[2] * p.scale_log2 : -INFINITY;
        float x3 = kh < end1 ? sacc[3] * p.scale_log2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);   // decode: finite, as key0 < k_end
        // extending, a row may have seen no key yet: keep a finite reference so that the
        // rescale and the weights below are 0 rather than NaN (2^-inf is +0 on the SFU)
        const float r0 = EXT && n0 == -INFINITY ? 0.f : n0, r1 = EXT && n1 == -INFINITY ? 0.f : n1;
        const float a0 = fast_exp2(m0 - r0), a1 = fast_exp2(m1 - r1);
        const float p0 = fast_exp2(x0 - r0), p1 = fast_exp2(x1 - r1), p2 = fast_exp2(x2 - r0), p3 = fast_exp2(x3 - r1);
        l0 = l0 * a0 + p0 + p2;
        l1 = l1 * a1 + p1 + p3;
        m0 = n0;
        m1 = n1;
        // the accumulators change only where a running maximum moved (most stages, once the
        // first keys are in, move none: then the warp skips the multiplies)
        if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                o[i][0] *= a0;
                o[i][1] *= a1;
                o[i][2] *= a0;
                o[i][3] *= a1;
            }
        }
        const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
        {
            const int mi = lane >> 3, rr = lane & 7;
            const int vrow = warp * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                uint32_t a[4];
                const int ch = 2 * i + (mi & 1);
                ldmatrix_x4_trans(vbuf(st) + (uint32_t)(vrow * ROWB) + swz(vrow, ch) * 16, a[0], a[1], a[2], a[3]);
                mma_bf16_16816(o[i], a, pb0, pb1);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();   // all warps done with the ring: reuse it for the cross-warp merge

    // Row sums across the 8 lanes sharing t4.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    // rows padded to D + 4 floats: the four lanes of a quad (t4) store rows 2*t4 (+1) of the
    // same columns, which a D-float row stride would put in one bank
    constexpr int RS = D + 4;
    float* red_o = reinterpret_cast<float*>(smem);                 // [4 warps][8 rows][RS]
    float* red_ml = red_o + 4 * 8 * RS;                            // [4 warps][8 rows][2]
    float* red_w = red_ml + 4 * 8 * 2;                             // [4 warps][8 rows]
    float* row_lse = red_w + 4 * 8;                                // [8 rows] (log2 domain)
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        const int d = 16 * i + r8;
        red_o[(warp * 8 + 2 * t4) * RS + d] = o[i][0];
        red_o[(warp * 8 + 2 * t4 + 1) * RS + d] = o[i][1];
        red_o[(warp * 8 + 2 * t4) * RS + d + 8] = o[i][2];
        red_o[(warp * 8 + 2 * t4 + 1) * RS + d + 8] = o[i][3];
    }
    if (r8 == 0) {
        red_ml[(warp * 8 + 2 * t4) * 2 + 0] = m0;
        red_ml[(warp * 8 + 2 * t4) * 2 + 1] = l0;
        red_ml[(warp * 8 + 2 * t4 + 1) * 2 + 0] = m1;
        red_ml[(warp * 8 + 2 * t4 + 1) * 2 + 1] = l1;
    }
    __syncthreads();
    // each row's merge weights, once: warp w's part counts 2^(m_w - M) / L, where M is the
    // largest running maximum and L = sum_w 2^(m_w - M) l_w
    if (tid < 8) {
        const int n = tid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, red_ml[(w * 8 + n) * 2]);
        float sc[4], L = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float mw = red_ml[(w * 8 + n) * 2];
            sc[w] = mw == -INFINITY ? 0.f : exp2f(mw - M);
            L += sc[w] * red_ml[(w * 8 + n) * 2 + 1];
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int w = 0; w < 4; ++w) red_w[w * 8 + n] = sc[w] * inv;
        row_lse[n] = M + log2f(L);
    }
    __syncthreads();
    constexpr int HALF = D / 2;                                    // two dims per thread and pass
    for (int idx = tid; idx < nrows * HALF; idx += DEC_THREADS) {
        const int n = idx / HALF, d = 2 * (idx - n * HALF);
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float wt = red_w[w * 8 + n];
            const float2 v = *reinterpret_cast<const float2*>(red_o + (w * 8 + n) * RS + d);
            acc0 += wt * v.x;
            acc1 += wt * v.y;
        }
        const int64_t slot = rows.out_row(n);
        if (EXT) {
            __nv_bfloat16* dst = ext.out + slot * D + d;
            if (ext.pair_store) {
                *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc0, acc1);
            } else {
                dst[0] = __float2bfloat16_rn(acc0);
                dst[1] = __float2bfloat16_rn(acc1);
            }
            if (d == 0 && ext.lse) ext.lse[slot] = row_lse[n] * LN2;
        } else {
            *reinterpret_cast<float2*>(p.part_o + slot * D + d) = make_float2(acc0, acc1);
            if (d == 0) p.part_lse[slot] = row_lse[n];
        }
    }
    __syncthreads();
}

// Private chunks: blockIdx = (chunk, kv head, request).  Keys [shared_len_b + c*chunk, ...).
template <int D>
__global__ void __launch_bounds__(DEC_THREADS) decode_private_kernel(DecodeParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int32_t L = p.kv_lens[b];
    const int shared = p.shared_of ? p.shared_of[b] : 0;   // loaded together with L
    if (L < 1 || L > p.max_len || L > p.stride) {
        if (c == 0 && g == 0 && threadIdx.x == 0) report(p.status, RX_DEV_BAD_LENGTH);
        return;
    }
    const int k_begin = shared + c * p.chunk;
    if (k_begin >= L) return;
    const int k_end = min(L, k_begin + p.chunk);
    const DecRowMap rows{(int64_t)b * p.hq + (int64_t)g * p.group, (int64_t)p.max_chunks + p.grp_chunks, c};
    dec_chunk<D>(p, p.r2t + (int64_t)b * p.stride, k_begin, k_end, g, rows, p.group, smem,
                 reinterpret_cast<int32_t*>(smem + dec_ring_bytes(D)));
}

// Small extend: blockIdx = (kv head, request).  A request's n_b new tokens times the query
// heads of a kv head (<= 8 rows) attend causally over all of its P_b + n_b keys in one
// chunk, and write the final output rows.
template <int D>
__global__ void __launch_bounds__(DEC_THREADS) extend_small_kernel(DecodeParams p, const int64_t* qo_indptr,
                                                                   const int32_t* prefix_lens, int32_t max_qo_len,
                                                                   __nv_bfloat16* out, float* lse, int pair_store) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int g = blockIdx.x, b = blockIdx.y;
    // Launched with programmatic serialization: the block may start while the kernel before it
    // in the stream (kv_pool_write, in a step) finishes, and waits for that kernel before it
    // reads anything (in a step, the offsets, the lengths and the table are all its output).
    pdl_wait();
    // The request's slot-table row is loaded first, up to the table's stride (a launch
    // parameter): its loads are in flight together with the request's offsets instead of
    // waiting for them (one dependent round trip fewer before the first K/V stage).
    int32_t* slot_s = reinterpret_cast<int32_t*>(smem + dec_ring_bytes(D));
    constexpr int PRE = DEC_MAX_CHUNK / DEC_THREADS;
    const int lim = (int)min(p.stride, (int64_t)DEC_MAX_CHUNK);
    const int32_t* row = p.r2t + (int64_t)b * p.stride;
    int32_t pre[PRE];
#pragma unroll
    for (int u = 0; u < PRE; ++u) {
        const int i = (int)threadIdx.x + u * DEC_THREADS;
        pre[u] = i < lim ? row[i] : -1;
    }
    const int64_t qo0 = qo_indptr[b];
    const int n = (int)(qo_indptr[b + 1] - qo0);
    const int P = prefix_lens[b];
    if (n <= 0) return;
    if (n > max_qo_len || n * p.group > 8 || P < 0 || (int64_t)P + n > p.stride || P + n > DEC_MAX_CHUNK) {
        if (g == 0 && threadIdx.x == 0) report(p.status, RX_DEV_BAD_LENGTH);
        return;
    }
    // the staged list: checked slots for the request's P + n keys, -1 after them
#pragma unroll
    for (int u = 0; u < PRE; ++u) {
        const int i = (int)threadIdx.x + u * DEC_THREADS;
        slot_s[i] = i < P + n ? checked_slot(p, pre[u]) : -1;
    }
    const ExtRowMap rows{qo0, p.hq, g * p.group, p.group};
    ExtRows ext{P, p.group, out, lse, pair_store != 0};
    dec_chunk<D, true>(p, row, 0, P + n, g, rows, n * p.group, smem, slot_s, ext, true);
}

int launch_extend_small(const SmallExtendArgs& a, cudaStream_t stream) {
    DecodeParams p{};
    p.q = (const __nv_bfloat16*)a.q;
    p.r2t = a.r2t;
    p.stride = a.stride;
    p.k_pool = (const __nv_bfloat16*)a.k_pool;
    p.v_pool = (const __nv_bfloat16*)a.v_pool;
    p.num_slots = a.num_slots;
    p.batch = a.batch;
    p.hq = a.hq;
    p.hkv = a.hkv;
    p.group = a.hq / a.hkv;
    p.scale_log2 = a.scale * LOG2E;
    p.status = a.status;
    const int smem = dec_ring_bytes(a.head_dim) + DEC_MAX_CHUNK * 4;
    dim3 grid((unsigned)a.hkv, (unsigned)a.batch);
    static PerDeviceOnce attr[2];
    const int rc = per_device_once(attr[a.head_dim == 128 ? 1 : 0], [&] {
        const cudaError_t e =
            a.head_dim == 128
                ? cudaFuncSetAttribute(extend_small_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                : cudaFuncSetAttribute(extend_small_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            set_error("prefix_extend_attention: cannot set the small-extend shared memory size: %s",
                      cudaGetErrorString(e));
            return (int)RX_ECUDA;
        }
        return (int)RX_OK;
    });
    if (rc != RX_OK) return rc;
    const int pair_store = ((uintptr_t)a.out & 3) == 0 ? 1 : 0;   // bf16 pairs in one store
    // programmatic serialization: the kernel may start while the kernel before it in the stream
    // (kv_pool_write, in a step) finishes, and waits for it before reading the table or pools
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(DEC_THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr_pdl[1];
    attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr_pdl;
    cfg.numAttrs = 1;
    cudaError_t e = a.head_dim == 128
                        ? cudaLaunchKernelEx(&cfg, extend_small_kernel<128>, p, a.qo_indptr, a.prefix_lens,
                                             (int32_t)a.max_qo_len, (__nv_bfloat16*)a.out, a.lse, pair_store)
                        : cudaLaunchKernelEx(&cfg, extend_small_kernel<64>, p, a.qo_indptr, a.prefix_lens,
                                             (int32_t)a.max_qo_len, (__nv_bfloat16*)a.out, a.lse, pair_store);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("prefix_extend_attention: small-extend launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

// Merge the private and shared partials of each (request, head): one warp per item.  The
// loads are laid out to overlap (length and group id together; one partial's lse per lane,
// reduced by shuffles; the partial rows four at a time): the kernel is a short chain of
// dependent global round trips, not a bandwidth problem.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(DecodeParams p, __nv_bfloat16* out, float* lse) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * 4 + warp;   // (request, head)
    if (item >= (int64_t)p.batch * p.hq) return;
    const int b = (int)(item / p.hq);
    const int32_t L = p.kv_lens[b];
    const int shared = p.shared_of ? p.shared_of[b] : 0;
    if (L < 1 || L > p.max_len || L > p.stride) return;
    const int npriv = (L - shared + p.chunk - 1) / p.chunk;
    const int n = npriv + (shared + p.chunk - 1) / p.chunk;   // private chunks, then shared ones
    const int per = p.max_chunks + p.grp_chunks;
    const float* po = p.part_o + item * per * D;
    const float* pl = p.part_lse + item * per;
    auto idx = [&](int s) { return s < npriv ? s : p.max_chunks + (s - npriv); };
    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, pl[idx(s)]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    constexpr int E = D / 32;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float W = 0.f;
#pragma unroll 4
    for (int s = 0; s < n; ++s) {
        const int i = idx(s);
        const float w = exp2f(pl[i] - M);
        W += w;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += w * po[(int64_t)i * D + lane + 32 * e];
    }
    __nv_bfloat16* orow = out + item * D;
#pragma unroll
    for (int e = 0; e < E; ++e) orow[lane + 32 * e] = __float2bfloat16_rn(acc[e] / W);
    if (lse && lane == 0) lse[item] = (M + log2f(W)) * LN2;
}

// Each request's count of shared keys (its group's shared run, cut to its own length; 0 outside
// every group), and each group's source slot-table row (its first member): one block, every
// request cleared before the groups' members are written.  The decode kernels then learn where
// a request's private keys start from one load, beside its length.
__global__ void __launch_bounds__(512) decode_group_map_kernel(DecodeParams p, int32_t* shared_of) {
    for (int b = threadIdx.x; b < p.batch; b += blockDim.x) shared_of[b] = 0;
    __syncthreads();
    for (int gid = threadIdx.x; gid < p.num_groups; gid += blockDim.x) p.group_src[gid] = p.grp_members[p.grp_indptr[gid]];
    const int n = p.num_groups > 0 ? p.grp_indptr[p.num_groups] : 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int lo = 0, hi = p.num_groups - 1;       // the group of member i
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.grp_indptr[mid] <= i) lo = mid; else hi = mid - 1;
        }
        const int b = p.grp_members[i];
        if (b >= 0 && b < p.batch) shared_of[b] = min(p.grp_len[lo], p.kv_lens[b]);
        else report(p.status, RX_DEV_BAD_LENGTH);
    }
}

// A side stream per device and two events: the shared-prefix part runs there, concurrently
// with the private part on the caller's stream (they only meet in the merge).
struct DecodeFork {
    cudaStream_t side = nullptr;
    cudaEvent_t ready = nullptr, shared_done = nullptr;
    std::mutex use;
};
static std::mutex g_fork_mu;
static std::unordered_map<int, DecodeFork> g_forks;

static DecodeFork* decode_fork() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_fork_mu);
    DecodeFork& f = g_forks[dev];
    if (!f.side) {
        if (cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.ready, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.shared_done, cudaEventDisableTiming) != cudaSuccess) {
            f.side = nullptr;
            return nullptr;
        }
    }
    return &f;
}

static int dec_chunk_keys(int32_t batch, int32_t hkv, int32_t max_kv_len) {
    // Long chunks amortise each CTA's start (slot staging, Q fragments) and end (cross-warp
    // merge, partial write) over more bytes; short ones keep enough CTAs to fill 152 SMs.
    auto ctas = [&](int c) { return (int64_t)batch * hkv * ((max_kv_len + c - 1) / c); };
    if (ctas(1024) >= 152 * 16) return 1024;
    if (ctas(512) >= 152 * 4) return 512;
    return 256;
}

struct DecodeLayout {
    int chunk, max_chunks, grp_chunks;
    size_t part_o_bytes, part_lse_bytes, shared_of_bytes, group_src_bytes, total;
};

static DecodeLayout dec_layout(const rx_attn_desc* d, int32_t batch, int32_t max_kv_len, const rx_shared_groups* grp) {
    DecodeLayout L{};
    L.chunk = dec_chunk_keys(batch, d->hkv, max_kv_len);
    L.max_chunks = (max_kv_len + L.chunk - 1) / L.chunk;
    L.grp_chunks = (grp && grp->num_groups > 0) ? (grp->max_group_len + L.chunk - 1) / L.chunk : 0;
    const size_t per = (size_t)(L.max_chunks + L.grp_chunks);
    L.part_o_bytes = (size_t)batch * d->hq * per * d->head_dim * sizeof(float);
    L.part_lse_bytes = (size_t)batch * d->hq * per * sizeof(float);
    L.shared_of_bytes = (grp && grp->num_groups > 0) ? (size_t)batch * sizeof(int32_t) : 0;
    L.group_src_bytes = (grp && grp->num_groups > 0) ? (size_t)grp->num_groups * sizeof(int32_t) : 0;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    L.total = up(L.part_o_bytes) + up(L.part_lse_bytes) + up(L.shared_of_bytes) + up(L.group_src_bytes);
    return L;
}

static size_t dec_smem_bytes(int D) { return (size_t)dec_ring_bytes(D) + DEC_MAX_CHUNK * sizeof(int32_t); }

}  // namespace rx

using namespace rx;

extern "C" size_t decode_workspace_bytes(const rx_attn_desc* desc, int32_t batch, int32_t max_kv_len,
                                         const rx_shared_groups* groups) {
    if (!desc || batch < 0 || max_kv_len < 1 || desc->hkv <= 0 || desc->hq <= 0) return 0;
    // the CUDA-core path (fp32, or more than 8 query heads per kv head) takes no workspace
    if (desc->dtype == RX_F32 || desc->hq / desc->hkv > 8) return 0;
    return dec_layout(desc, batch, max_kv_len, groups).total;
}

extern "C" int decode_attention(const rx_attn_desc* desc, int32_t batch, const void* d_q,
                                const int32_t* d_req_to_token, int64_t r2t_stride, const int32_t* d_kv_lens,
                                const rx_shared_groups* groups, const void* d_k_pool, const void* d_v_pool,
                                void* d_out, float* d_lse, int32_t max_kv_len, void* d_workspace,
                                size_t ws_bytes, int32_t* d_status, void* stream_) {
    RX_TRACE("decode_attention");
    RX_REQUIRE(desc && batch >= 0 && max_kv_len >= 1 && r2t_stride >= 0, "decode_attention: bad arguments");
    RX_REQUIRE(desc->hq > 0 && desc->hkv > 0 && desc->hq % desc->hkv == 0, "decode_attention: bad head counts");
    RX_REQUIRE(desc->head_dim == 64 || desc->head_dim == 128, "decode_attention: head_dim must be 64 or 128");
    if (batch == 0) return RX_OK;
    RX_REQUIRE(d_q && d_req_to_token && d_kv_lens && d_k_pool && d_v_pool && d_out,
               "decode_attention: null device pointer");
    cudaStream_t stream = (cudaStream_t)stream_;
    const int group = desc->hq / desc->hkv;
    if (desc->dtype == RX_F32 || group > 8) {
        // CUDA-core path: fp32 (exact arithmetic of the tiny workload) or > 8 heads per kv head.
        SimtParams sp{};
        sp.batch = batch;
        sp.hq = desc->hq;
        sp.hkv = desc->hkv;
        sp.total_rows = batch;
        sp.q = d_q;
        sp.kv_lens = d_kv_lens;
        sp.r2t = d_req_to_token;
        sp.stride = r2t_stride;
        sp.k_pool = d_k_pool;
        sp.v_pool = d_v_pool;
        sp.num_slots = desc->num_slots;
        sp.out = d_out;
        sp.lse = d_lse;
        sp.scale = desc->scale;
        sp.max_len = max_kv_len;
        sp.status = d_status;
        return launch_attn_simt(sp, desc->dtype, desc->head_dim, stream);
    }
    RX_REQUIRE(desc->dtype == RX_BF16, "decode_attention: unknown dtype %d", desc->dtype);
    const bool use_groups = groups && groups->num_groups > 0;
    if (use_groups)
        RX_REQUIRE(groups->d_group_indptr && groups->d_group_members && groups->d_group_len &&
                       groups->max_group_size >= 1 && groups->max_group_len >= 1,
                   "decode_attention: incomplete shared groups");
    const DecodeLayout lay = dec_layout(desc, batch, max_kv_len, use_groups ? groups : nullptr);
    RX_REQUIRE(d_workspace && ws_bytes >= lay.total, "decode_attention: workspace of %zu bytes, %zu needed",
               ws_bytes, lay.total);
    RX_REQUIRE(((uintptr_t)d_workspace & 255) == 0, "decode_attention: workspace must be 256-byte aligned");
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    unsigned char* ws = (unsigned char*)d_workspace;
    DecodeParams p{};
    p.q = (const __nv_bfloat16*)d_q;
    p.r2t = d_req_to_token;
    p.stride = r2t_stride;
    p.kv_lens = d_kv_lens;
    p.k_pool = (const __nv_bfloat16*)d_k_pool;
    p.v_pool = (const __nv_bfloat16*)d_v_pool;
    p.num_slots = desc->num_slots;
    p.batch = batch;
    p.hq = desc->hq;
    p.hkv = desc->hkv;
    p.group = group;
    p.scale_log2 = desc->scale * LOG2E;
    p.chunk = lay.chunk;
    p.max_chunks = lay.max_chunks;
    p.max_len = max_kv_len;
    p.part_o = (float*)ws;
    p.part_lse = (float*)(ws + up(lay.part_o_bytes));
    p.status = d_status;
    p.grp_chunks = lay.grp_chunks;
    int32_t* shared_of = nullptr;
    if (use_groups) {
        shared_of = (int32_t*)(ws + up(lay.part_o_bytes) + up(lay.part_lse_bytes));
        p.group_src = (int32_t*)(ws + up(lay.part_o_bytes) + up(lay.part_lse_bytes) + up(lay.shared_of_bytes));
        p.num_groups = groups->num_groups;
        p.grp_indptr = groups->d_group_indptr;
        p.grp_members = groups->d_group_members;
        p.grp_len = groups->d_group_len;
        p.grp_rows_max = groups->max_group_size * group;
        p.shared_of = shared_of;
    }
    const int D = desc->head_dim;
    const size_t smem = dec_smem_bytes(D);
    static PerDeviceOnce attr_set[2];
    const int arc = per_device_once(attr_set[D == 128 ? 1 : 0], [&] {
        const cudaError_t e1 =
            D == 128 ? cudaFuncSetAttribute(decode_private_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                     : cudaFuncSetAttribute(decode_private_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e1 == cudaSuccess)   // the whole unified L1 as shared memory: three CTAs per SM
            (void)(D == 128 ? cudaFuncSetAttribute(decode_private_kernel<128>, cudaFuncAttributePreferredSharedMemoryCarveout, 100)
                            : cudaFuncSetAttribute(decode_private_kernel<64>, cudaFuncAttributePreferredSharedMemoryCarveout, 100));
        if (e1 != cudaSuccess) {
            set_error("decode_attention: cannot set shared memory size: %s", cudaGetErrorString(e1));
            return (int)RX_ECUDA;
        }
        return (int)RX_OK;
    });
    if (arc != RX_OK) return arc;
    dim3 grid((unsigned)lay.max_chunks, (unsigned)desc->hkv, (unsigned)batch);
    auto launch_private = [&] {
        if (D == 128) decode_private_kernel<128><<<grid, DEC_THREADS, smem, stream>>>(p);
        else decode_private_kernel<64><<<grid, DEC_THREADS, smem, stream>>>(p);
    };
    DecodeFork* fork = nullptr;
    std::unique_lock<std::mutex> fork_lock;
    if (use_groups) {
        decode_group_map_kernel<<<1, 512, 0, stream>>>(p, shared_of);
        // The shared runs go through the tcgen05 kernel: a group's stacked query rows read
        // each shared K/V row once per 256 rows.  On the side stream, concurrently with the
        // private part (both need only the group map); the merge waits for both.
        fork = decode_fork();
        cudaStream_t shared_stream = stream;
        if (fork) {
            fork_lock = std::unique_lock<std::mutex>(fork->use);
            if (cudaEventRecord(fork->ready, stream) == cudaSuccess &&
                cudaStreamWaitEvent(fork->side, fork->ready, 0) == cudaSuccess)
                shared_stream = fork->side;
            else
                fork = nullptr;
        }
        // The private part is launched first: its CTAs fill the GPU at once, and the shared
        // part's CTAs (a whole SM each) take SMs as the private part's last wave drains,
        // instead of holding SMs from the private part's start.
        launch_private();
        SharedTcParams sp{};
        sp.q = d_q;
        sp.r2t = d_req_to_token;
        sp.stride = r2t_stride;
        sp.k_pool = d_k_pool;
        sp.v_pool = d_v_pool;
        sp.num_slots = desc->num_slots;
        sp.batch = batch;
        sp.hq = desc->hq;
        sp.hkv = desc->hkv;
        sp.head_dim = D;
        sp.scale = desc->scale;
        sp.status = d_status;
        sp.num_groups = groups->num_groups;
        sp.max_group_rows = groups->max_group_size;     // one query row per member in decode
        sp.grp_row_indptr = groups->d_group_indptr;
        sp.grp_rows = groups->d_group_members;
        sp.grp_src = p.group_src;
        sp.grp_len = groups->d_group_len;
        sp.chunk = lay.chunk;
        sp.n_chunks = lay.grp_chunks;
        sp.part_o = p.part_o;
        sp.part_lse = p.part_lse;
        sp.part_per = lay.max_chunks + lay.grp_chunks;
        sp.part_base = lay.max_chunks;
        const int rc = launch_shared_prefix_tc(sp, shared_stream);
        if (rc != RX_OK) return rc;
        if (fork && cudaEventRecord(fork->shared_done, fork->side) != cudaSuccess) {
            set_error("decode_attention: cannot record the shared part's event");
            return RX_ECUDA;
        }
    }
    if (!use_groups) launch_private();
    if (fork && cudaStreamWaitEvent(stream, fork->shared_done, 0) != cudaSuccess) {
        set_error("decode_attention: cannot join the shared part");
        return RX_ECUDA;
    }
    const int64_t items = (int64_t)batch * desc->hq;
    const unsigned mblocks = (unsigned)((items + 3) / 4);
    if (D == 128) decode_merge_kernel<128><<<mblocks, 128, 0, stream>>>(p, (__nv_bfloat16*)d_out, d_lse);
    else decode_merge_kernel<64><<<mblocks, 128, 0, stream>>>(p, (__nv_bfloat16*)d_out, d_lse);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("decode_attention: launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

// ----------------------------------------------------------------------------------------
// decode_attention_noalloc: decode_attention with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory per call: a plug-in running inside a host
// application whose allocator has already reserved the GPU's memory (a raw cudaMalloc would
// fail or bypass the host's accounting), a serving loop that must not stall on
// cudaMalloc/cudaFree (both may synchronise the device), or a plain C caller with no
// allocator of its own to provide the split-KV workspace.  For them this entry point keeps
// the workspace in one file-scope device array of RX_DECODE_NOALLOC_SCRATCH_BYTES, which
// every GPU that loads the library holds until the process exits.  Host code cannot use
// the array's name as a device address: every call looks the address up with
// cudaGetSymbolAddress on the current device (a host-side lookup; the device code is loaded
// on a device's first call), so the address follows the current context, also after a
// cudaDeviceReset.
namespace rx {

static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[RX_DECODE_NOALLOC_SCRATCH_BYTES];

}  // namespace rx

extern "C" int decode_attention_noalloc(const rx_attn_desc* desc, int32_t batch, const void* d_q,
                                        const int32_t* d_req_to_token, int64_t r2t_stride,
                                        const int32_t* d_kv_lens, const rx_shared_groups* groups,
                                        const void* d_k_pool, const void* d_v_pool, void* d_out, float* d_lse,
                                        int32_t max_kv_len, int32_t* d_status, void* stream) {
    RX_TRACE("decode_attention_noalloc");
    RX_REQUIRE(desc && batch >= 0 && max_kv_len >= 1, "decode_attention_noalloc: bad arguments");
    if (batch == 0) return RX_OK;
    const size_t need = decode_workspace_bytes(desc, batch, max_kv_len, groups);
    RX_REQUIRE(need <= (size_t)RX_DECODE_NOALLOC_SCRATCH_BYTES,
               "decode_attention_noalloc: this batch needs %zu bytes of scratch, the static scratch holds %zu "
               "(use decode_attention with a caller-provided workspace, or split the batch)",
               need, (size_t)RX_DECODE_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&scratch, g_decode_noalloc_scratch);
    if (e != cudaSuccess || !scratch) {
        set_error("decode_attention_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    // The split-KV partials and the group map are fully written before they are read in
    // every call, so the scratch needs no clearing between calls.
    return decode_attention(desc, batch, d_q, d_req_to_token, r2t_stride, d_kv_lens, groups, d_k_pool, d_v_pool,
                            d_out, d_lse, max_kv_len, scratch, (size_t)RX_DECODE_NOALLOC_SCRATCH_BYTES, d_status,
                            stream);
}
