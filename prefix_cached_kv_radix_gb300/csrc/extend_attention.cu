// Extend (prefill over new tokens) attention with a radix-cached prefix, on tcgen05 tensor
// cores with TMEM accumulators (sm_103a).
//
// "Prompt Caching" (Ultralytics glossary), "How prompt caching works": on a cache hit only
// the new tokens run through the model; because attention is causal, the cached prefix's
// keys/values (computed once, shared) stand in for recomputing it.  Row i of request b
// (position p = P_b + i) attends keys 0..p: the prefix gathered from scattered pool slots
// through req_to_token, then the request's own new tokens causally (self included).
// "SGLang: Efficient Execution of Structured Language Model Programs", RadixAttention:
// the prefix's KV is reused across requests rather than recomputed.
//
// GB300 design.  The work items are (request, kv head, 256 packed query rows): the query
// heads of a kv head (GQA group) are packed with the tokens, head fastest: packed row R ->
// token R / G, head g*G + R % G, so every K/V tile feeds G heads and the tile stays a dense
// contraction.  Two 128-row Q tiles share each K/V tile of 128 keys.  The grid is persistent:
// one CTA per SM, its rings, barriers and TMEM running on across items, so an item's set-up and
// output overlap the neighbouring items' work instead of each CTA starting and draining on its
// own.  The CTAs take the items in order from a per-stream work counter (the Q warp fetches the
// next item and hands its id to the other roles through a small ring in shared memory), so the
// items in flight stay a compact window whose K/V the L2 holds.  Roles (512 threads, four
// warpgroups, registers split 88 / 168 / 168 / 88 with setmaxnreg):
//   warp 0     Q loads: per item, once the previous item's last S has read a Q buffer, the
//              full 128-row tiles by TMA (one box per 64 columns, q seen as [token][head][D],
//              box 64 x G x 128/G, 128-byte swizzle), a ragged tile and every tile of the
//              shared-prefix mode row by row.
//   warps 1-3, 13-15  K/V loaders: 16-byte cp.async gathers of K and V tiles through the slot
//              table into separate K (3-deep) and V (2-deep) rings in the 128B-swizzled layouts
//              tcgen05 reads, on across item boundaries.  Each thread's arrival on a tile's full
//              barrier is made by the copy hardware when its copies land
//              (cp.async.mbarrier.arrive), so loaders wait only for free slots; slot ids are
//              prefetched a tile ahead.
//   warp 12    TMEM allocator and single-thread tcgen05.mma issuer, per K/V tile j and
//              Q tile t:  O_t += P_t(j) V(j)  (M=128, N=D, K=128, P from TMEM, in two halves of
//              64 keys as the softmax publishes them), then at once
//              S_t(j+1) = Q_t K(j+1)^T  (M=128, N=128, K=D) into the same TMEM columns -- the
//              tensor pipe runs one thread's MMAs in order, so P is read before it is
//              overwritten.  Completion via tcgen05.commit; after an item's last PV on a tile a
//              commit tells the softmax warps its O is complete.
//   warps 4-7  softmax of Q tile 0; warps 8-11 softmax of Q tile 1: tcgen05.ld of a score
//              row per thread, causal mask, online softmax in the exp2 domain with a lazy
//              rescale (the reference max only moves when the row max grows by more than
//              2^8, which keeps every P <= 256), P packed to bf16 and stored over the row's
//              scores in TMEM (tcgen05.st) in two halves, each released to the tensor core at
//              once; fp32 pairs use the packed f32x2 forms.  At an item's end each thread
//              writes its normalised row straight from TMEM while the tensor core already
//              works on the next item's scores.
// TMEM columns: S0/P0 [0,128) S1/P1 [128,256) O0 [256,256+D) O1 after.  While one Q tile's
// softmax runs, the tensor core works on the other's GEMMs.  Every wait is bounded; on
// time-out the kernel records RX_DEV_TIMEOUT, drains its async copies, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "radix_attn.h"
#include "rx_common.h"
#include "rx_device.cuh"
#include "rx_kernels.h"

namespace rx {

constexpr int EXT_BN = 128;       // keys per K/V tile
constexpr int EXT_THREADS = 512;  // 16 warps
constexpr int EXT_MMA_WARP = 12;
constexpr int EXT_Q_WARP = 0;      // loads every item's Q tiles (TMA, or row gathers for ragged tiles)
constexpr int EXT_LOADERS = 192;  // K/V gathers: warps 1-3 and 13-15
constexpr int EXT_RING = 4;        // items handed from the Q warp to the other roles, in flight
// warps that take items from the ring besides the Q warp that fills it: six loader warps, the
// MMA warp and eight softmax warps (one arrival each per item)
constexpr int EXT_ITEM_CONSUMERS = 15;
constexpr uint32_t EXT_REGS_SOFTMAX = 168, EXT_REGS_OTHER = 88;   // 2*128*88 + 2*128*168 = 512*128
constexpr float EXT_LOG2E = 1.4426950408889634f;
constexpr float EXT_LN2 = 0.6931471805599453f;
constexpr float EXT_RESCALE_THRESHOLD = 8.0f;   // log2 units

struct ExtendParams {
    const __nv_bfloat16* q;
    const int64_t* qo_indptr;
    const int32_t* prefix_lens;
    const int32_t* r2t;
    int64_t stride;
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    int64_t num_slots;
    __nv_bfloat16* out;
    float* lse;
    int32_t batch, hq, hkv, group;
    float scale_log2;
    int32_t max_qo_len;
    int32_t* status;
    // Shared-prefix mode: CTA (row tile * n_chunks + chunk, kv head, group).  The rows of
    // group gid are the query rows grp_rows[grp_row_indptr[gid] ..] (global row ids of q,
    // head fastest within a row); keys are one chunk of the group's shared run, taken from
    // the slot-table row grp_src[gid], unmasked; outputs are fp32 normalised partials and
    // log2-domain log-sum-exp at partial index part_base + chunk of (row, head).
    int32_t shared_mode;
    const int32_t* grp_row_indptr;
    const int32_t* grp_rows;
    const int32_t* grp_src;
    const int32_t* grp_len;
    int32_t chunk, n_chunks;
    float* part_o;
    float* part_lse;
    int32_t part_per, part_base;
    // Extend mode: tiled tensor map of q seen as [rows][hq][D] (box 64 x G x 128/G elements,
    // 128-byte swizzle), set by the host when G divides 128 and the buffer allows it.  Full
    // 128-row Q tiles are then loaded by TMA.
    int32_t q_map_ok;
    CUtensorMap q_map;
    // Persistent grid: the work items are the cells (x, kv head, request or group) of a
    // grid_x x hkv x (batch or groups) grid, x fastest.  With `work` (two counters: the next
    // item, and the CTAs done; zero at launch) the CTAs take items in order as they free up, so
    // the items in flight stay a compact window and share L2 (one CTA per item of the window
    // touches the same requests' K/V); without it CTA c takes items c, c + gridDim.x, ...
    int32_t grid_x, n_items;
    unsigned int* work;
};

template <int D>
struct ExtLayout {
    static constexpr int NK = D == 128 ? 3 : 4;    // K ring depth
    static constexpr int NV = D == 128 ? 2 : 4;    // V ring depth
    static constexpr int Q_TILE = 128 * D * 2;
    static constexpr int KV_TILE = EXT_BN * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * Q_TILE;
    static constexpr int OFF_V = OFF_K + NK * KV_TILE;
    static constexpr int OFF_BAR = OFF_V + NV * KV_TILE;
    // q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[2], p_full[half][2],
    // q_empty[2], o_ready[2], mma_done
    static constexpr int BAR_Q = 0, BAR_KF = 1, BAR_KE = 1 + NK, BAR_VF = 1 + 2 * NK, BAR_VE = 1 + 2 * NK + NV,
                         BAR_S = 1 + 2 * NK + 2 * NV, BAR_P = BAR_S + 2, BAR_QE = BAR_P + 4, BAR_OR = BAR_QE + 2,
                         BAR_IF = BAR_OR + 2, BAR_IE = BAR_IF + EXT_RING, BAR_DONE = BAR_IE + EXT_RING,
                         NBAR = BAR_DONE + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16 + 4 * EXT_RING;   // TMEM address, abort flag, item ring
    static constexpr int ALLOC = BYTES + 1024;   // room to align the base to 1024 B
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_O0 = 256;
    static constexpr int CPR = D / 8;                                   // 16-byte chunks per row
    static constexpr int NX = (EXT_BN * CPR + EXT_LOADERS - 1) / EXT_LOADERS;   // chunks per loader thread per tile
    static_assert(ALLOC <= 232448, "shared memory budget");
};

// One work item: a CTA's worth of rows of the grid (x, y, z) the kernel was written for.
// Extend: packed row R -> token R / G of request b (position P_b + R / G), head g*G + R % G.
// Shared-prefix: packed row R -> member R / G of group gid, head g*G + R % G, all keys.
struct ExtItem {
    bool valid;
    int g, b, n_b, P_b, rows_total, row0, kv_end, m0, x, ntiles, nkv;
    int64_t qo0;
    bool map_rows;
    const int32_t* slots_row;
};

// Decodes item index `it` (x fastest, then kv head, then request or group) and checks its
// lengths; an item with no rows, or with a length the table cannot hold (reported once per
// request or group, by its first item's thread 0), is not valid.  Every role of the CTA
// decodes the same items in the same order, so they agree on which are skipped.
__device__ __forceinline__ ExtItem ext_item(const ExtendParams& p, int it) {
    ExtItem r{};
    const int gx = p.grid_x;
    r.x = it % gx;
    r.g = (it / gx) % p.hkv;
    const int z = it / (gx * p.hkv);
    const int G = p.group;
    r.valid = false;
    if (!p.shared_mode) {
        r.b = z;
        r.qo0 = p.qo_indptr[r.b];
        r.n_b = (int)(p.qo_indptr[r.b + 1] - r.qo0);
        r.P_b = p.prefix_lens[r.b];
        r.rows_total = r.n_b * G;
        r.row0 = r.x * 256;
        if (r.row0 >= r.rows_total || r.n_b <= 0) return r;
        if (r.n_b > p.max_qo_len || r.P_b < 0 || (int64_t)r.P_b + r.n_b > p.stride) {
            if (threadIdx.x == 0 && r.x == 0 && r.g == 0) report(p.status, RX_DEV_BAD_LENGTH);
            return r;
        }
        const int last_row = min(r.row0 + 256, r.rows_total) - 1;
        r.kv_end = r.P_b + last_row / G + 1;              // keys needed by this item
        r.slots_row = p.r2t + (int64_t)r.b * p.stride;
    } else {
        const int gid = z;
        const int c = r.x % p.n_chunks;
        r.m0 = p.grp_row_indptr[gid];
        r.rows_total = (p.grp_row_indptr[gid + 1] - r.m0) * G;
        r.row0 = (r.x / p.n_chunks) * 256;
        const int len = p.grp_len[gid];
        const int k_lo = c * p.chunk;
        if (r.row0 >= r.rows_total || k_lo >= len) return r;
        if (len > p.stride) {
            if (threadIdx.x == 0 && r.x == 0 && r.g == 0) report(p.status, RX_DEV_BAD_LENGTH);
            return r;
        }
        r.kv_end = min(len, k_lo + p.chunk) - k_lo;       // keys of this chunk, relative to k_lo
        r.slots_row = p.r2t + (int64_t)p.grp_src[gid] * p.stride + k_lo;
    }
    r.ntiles = r.rows_total - r.row0 > 128 ? 2 : 1;
    // full tiles of the extend mode go through the tensor map (token coordinates are 31-bit)
    r.map_rows = !p.shared_mode && r.qo0 + r.n_b <= INT32_MAX;
    r.nkv = (r.kv_end + EXT_BN - 1) / EXT_BN;
    r.valid = true;
    return r;
}

template <int D>
__global__ void __launch_bounds__(EXT_THREADS, 1) extend_tc_kernel(const __grid_constant__ ExtendParams p) {
    using LY = ExtLayout<D>;
    constexpr int CPR = LY::CPR;
    constexpr int NX = LY::NX;
    constexpr int NK = LY::NK;
    constexpr int NV = LY::NV;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + LY::OFF_BAR;
    auto bar = [&](int i) { return bar0 + (uint32_t)(8 * i); };
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(gbase + LY::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + LY::OFF_MISC + 4);
    volatile int32_t* item_ring = reinterpret_cast<volatile int32_t*>(gbase + LY::OFF_MISC + 16);
    // This CTA's k-th item (-1: none left).  Round-robin without a work counter; with one, the
    // entry the Q warp wrote into the ring (a whole warp waits; lane 0 releases the entry).
    auto take_item_warp = [&](int k) -> int {
        if (!p.work) {
            const int64_t it = (int64_t)blockIdx.x + (int64_t)k * gridDim.x;
            return it < p.n_items ? (int)it : -1;
        }
        const int e = k % EXT_RING;
        if (!warp_wait(bar(LY::BAR_IF + e), (k / EXT_RING) & 1, abort_flag, p.status)) return -1;
        const int item = item_ring[e];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(bar(LY::BAR_IE + e));
        return item;
    };
    // the same for the single MMA-issuing thread
    auto take_item_thread = [&](int k) -> int {
        if (!p.work) {
            const int64_t it = (int64_t)blockIdx.x + (int64_t)k * gridDim.x;
            return it < p.n_items ? (int)it : -1;
        }
        const int e = k % EXT_RING;
        if (!mbar_wait(bar(LY::BAR_IF + e), (k / EXT_RING) & 1, abort_flag, p.status)) return -1;
        const int item = item_ring[e];
        mbar_arrive(bar(LY::BAR_IE + e));
        return item;
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    // query row pointer of packed row R of an item (clamped to its last valid row by the caller)
    auto q_row = [&](int64_t qo0, int m0, int gh, int R) -> const __nv_bfloat16* {
        if (!p.shared_mode) return p.q + ((qo0 + R / G) * p.hq + gh * G + R % G) * D;
        return p.q + ((int64_t)p.grp_rows[m0 + R / G] * p.hq + gh * G + R % G) * D;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(LY::BAR_Q), 32 + 1);   // per item: the Q warp's lanes + lane 0's expect-tx arrival
        for (int i = 0; i < NK; ++i) {
            mbar_init(bar(LY::BAR_KF + i), EXT_LOADERS);
            mbar_init(bar(LY::BAR_KE + i), 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(bar(LY::BAR_VF + i), EXT_LOADERS);
            mbar_init(bar(LY::BAR_VE + i), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(LY::BAR_S + t), 1);
            mbar_init(bar(LY::BAR_P + t), 4);          // one arrival per softmax warp, keys 0-63
            mbar_init(bar(LY::BAR_P + 2 + t), 4);      // keys 64-127
            mbar_init(bar(LY::BAR_QE + t), 1);         // Q buffer t read by its item's last S
            mbar_init(bar(LY::BAR_OR + t), 1);         // O_t of an item complete
        }
        for (int i = 0; i < EXT_RING; ++i) {
            mbar_init(bar(LY::BAR_IF + i), 1);                        // entry i written
            mbar_init(bar(LY::BAR_IE + i), EXT_ITEM_CONSUMERS);       // entry i read by every role
        }
        mbar_init(bar(LY::BAR_DONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == EXT_MMA_WARP) {
        tmem_alloc(base + LY::OFF_MISC, LY::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int wg = warp >> 2;

    // Role dispatch on the warpgroup first, so that each register re-split dominates the
    // code that relies on it (the compiler allocates each region to its own limit).
    if (wg == 0 || wg == 3) {
    regs_decrease<EXT_REGS_OTHER>();
    if (warp != EXT_MMA_WARP) {
        if (warp == EXT_Q_WARP) {
        // ------------------------------------------------------------ Q loads
        // Per item: each Q buffer is refilled once the previous item that used it has had its
        // last S read it; full 128-row tiles of the extend mode by TMA (lane 0, one box per 64
        // columns, in the swizzled layout the MMA reads), a ragged last tile and every tile of
        // the shared-prefix mode row by row (rows past the end clamped to the last one).  A
        // warp of its own, so that the K/V loaders run on into the next item meanwhile.
        const uint32_t qs = base + LY::OFF_Q;
        int quse0 = 0, quse1 = 0;         // items so far that used Q buffer 0 / 1
        for (int k = 0;; ++k) {
            // the next item: from the work counter into the ring (once every role has read the
            // entry it replaces), or round-robin
            int item;
            if (p.work) {
                const int e = k % EXT_RING;
                if (k >= EXT_RING && !warp_wait(bar(LY::BAR_IE + e), ((k / EXT_RING) - 1) & 1, abort_flag, p.status))
                    break;
                if (lane == 0) {
                    const unsigned t = atomicAdd(&p.work[0], 1u);
                    item = t < (unsigned)p.n_items ? (int)t : -1;
                    item_ring[e] = item;
                    mbar_arrive(bar(LY::BAR_IF + e));   // release: the entry is visible to the waiters
                }
                item = __shfl_sync(0xffffffffu, item, 0);
            } else {
                const int64_t it = (int64_t)blockIdx.x + (int64_t)k * gridDim.x;
                item = it < p.n_items ? (int)it : -1;
            }
            if (item < 0) break;
            const ExtItem it = ext_item(p, item);
            if (!it.valid) continue;
            if (quse0 > 0 && !warp_wait(bar(LY::BAR_QE), (quse0 - 1) & 1, abort_flag, p.status)) break;
            if (it.ntiles > 1 && quse1 > 0 && !warp_wait(bar(LY::BAR_QE + 1), (quse1 - 1) & 1, abort_flag, p.status))
                break;
            quse0 += 1;
            quse1 += it.ntiles > 1 ? 1 : 0;
            const int n_full_q = (p.q_map_ok && it.map_rows) ? min(it.ntiles, (it.rows_total - it.row0) >> 7) : 0;
            if (lane == 0) {
                fence_proxy_async_smem();     // earlier generic-proxy writes of the buffers first
                mbar_arrive_expect_tx(bar(LY::BAR_Q), (uint32_t)(n_full_q * LY::Q_TILE));
                const int tok0 = (int)(it.qo0 + it.row0 / G);
                for (int t = 0; t < n_full_q; ++t)
                    for (int h = 0; h < D / 64; ++h)
                        tma_load_3d(qs + (uint32_t)(t * LY::Q_TILE + h * 128 * 128), &p.q_map, h * 64, it.g * G,
                                    tok0 + t * (128 / G), bar(LY::BAR_Q));
            }
            // The rows the TMA does not bring, two lanes per row: the row's source is found once
            // (in the shared-prefix mode through the group's row list) and the pair copies
            // neighbouring 16-byte chunks, so every 32-byte sector is read whole.
            for (int rr = n_full_q * 128 + (lane >> 1); rr < it.ntiles * 128; rr += 16) {
                const int t = rr >> 7, r = rr & 127;
                const int R = min(it.row0 + rr, it.rows_total - 1);
                const __nv_bfloat16* src = q_row(it.qo0, it.m0, it.g, R);
                const uint32_t rowb = qs + (uint32_t)(t * LY::Q_TILE + r * 128);
#pragma unroll
                for (int k = 0; k < CPR / 2; ++k) {
                    const int c = 2 * k + (lane & 1);
                    cp_async_16(rowb + (uint32_t)((c >> 3) * 128 * 128 + (((c & 7) ^ (r & 7)) << 4)), src + c * 8, 16);
                }
            }
            cp_async_arrive_noinc(bar(LY::BAR_Q));   // arrives once this lane's Q copies land
        }
        cp_async_wait_all();
        } else {
        // ------------------------------------------------------------ K/V loaders
        const int lt = warp < 4 ? (int)threadIdx.x - 32 : (int)threadIdx.x - (EXT_MMA_WARP + 1) * 32 + 96;
        const uint32_t nslots = (uint32_t)min(p.num_slots, (int64_t)1 << 31);
        // This thread copies the same 16-byte chunk (lt % CPR) of every key row it handles
        // (EXT_LOADERS is a multiple of CPR): its pool addresses differ by slot * row pitch only.
        static_assert(EXT_LOADERS % CPR == 0, "loader chunk per thread");
        const uint32_t pitch = (uint32_t)(p.hkv * D * 2);
        int gt = 0;                       // K/V tiles gathered so far (all items): ring position
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = take_item_warp(k);
            if (item < 0) break;
            const ExtItem it = ext_item(p, item);
            if (!it.valid) continue;
            // Slot ids of one tile (this thread's keys), loaded a tile ahead: the loads of tile
            // j+1 are issued once tile j's copies are, and first read after the next ring wait.
            // A key inside the context whose id is outside [0, num_slots) is reported and, like a
            // key past the context, zero-filled.
            int32_t sl[NX];
            const int kv_end = it.kv_end, nkv = it.nkv;
            const int32_t* slots_row = it.slots_row;
            auto inside = [&](int j, int x) {
                const int q = lt + EXT_LOADERS * x;
                return q < EXT_BN * CPR && j * EXT_BN + q / CPR < kv_end;
            };
            auto load_slots = [&](int j) {
#pragma unroll
                for (int x = 0; x < NX; ++x)
                    sl[x] = inside(j, x) ? slots_row[j * EXT_BN + (lt + EXT_LOADERS * x) / CPR] : -1;
            };
            const char* kb = reinterpret_cast<const char*>(p.k_pool + (size_t)it.g * D + (lt % CPR) * 8);
            const char* vb = reinterpret_cast<const char*>(p.v_pool + (size_t)it.g * D + (lt % CPR) * 8);
            // Gather one K or V tile (zero fill where sl < 0); the full barrier gets this
            // thread's arrival when its copies have landed (cp.async.mbarrier.arrive), so a
            // loader never waits for its own copies, only for free ring slots.
            auto issue = [&](uint32_t buf, const char* pb, uint32_t full) {
#pragma unroll
                for (int x = 0; x < NX; ++x) {
                    const int q = lt + EXT_LOADERS * x;
                    if (q < EXT_BN * CPR) {
                        const int key = q / CPR, c = q % CPR;
                        const uint32_t so =
                            (uint32_t)((c >> 3) * EXT_BN * 128 + key * 128 + (((c & 7) ^ (key & 7)) << 4));
                        cp_async_16(buf + so, pb + (size_t)(uint32_t)max(sl[x], 0) * pitch, sl[x] >= 0 ? 16u : 0u);
                    }
                }
                cp_async_arrive_noinc(full);
            };
            load_slots(0);
            for (int j = 0; j < nkv; ++j) {
                const int u = gt + j;                 // ring position of this tile
                const int ks = u % NK, vs = u % NV;
                if (u >= NK && !warp_wait(bar(LY::BAR_KE + ks), ((u / NK) - 1) & 1, abort_flag, p.status)) { ok = false; break; }
                bool bad = false;
#pragma unroll
                for (int x = 0; x < NX; ++x) {
                    const bool in = inside(j, x), valid = (uint32_t)sl[x] < nslots;
                    bad |= in && !valid;
                    sl[x] = (in && valid) ? sl[x] : -1;
                }
                if (bad) report(p.status, RX_DEV_BAD_SLOT);
                issue(base + LY::OFF_K + ks * LY::KV_TILE, kb, bar(LY::BAR_KF + ks));
                if (u >= NV && !warp_wait(bar(LY::BAR_VE + vs), ((u / NV) - 1) & 1, abort_flag, p.status)) { ok = false; break; }
                issue(base + LY::OFF_V + vs * LY::KV_TILE, vb, bar(LY::BAR_VF + vs));
                if (j + 1 < nkv) load_slots(j + 1);
            }
            gt += nkv;
        }
        cp_async_wait_all();                   // no copy may still be landing at teardown
        }
    } else {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(128, EXT_BN, 0, 0);
            constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 0, 1);
            const uint64_t qd0 = sdesc_sw128(base + LY::OFF_Q, 16, 1024);
            const uint64_t kd0 = sdesc_sw128(base + LY::OFF_K, 16, 1024);
            const uint64_t vd0 = sdesc_sw128(base + LY::OFF_V, EXT_BN * 128, 1024);
            // descriptor start addresses advance in 16-byte units in the low bits
            auto issue_s = [&](int t, int ks) {
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    umma_f16_ss(tmem + t * EXT_BN,
                                qd0 + (uint64_t)((t * LY::Q_TILE + (s >> 2) * 128 * 128 + (s & 3) * 32) >> 4),
                                kd0 + (uint64_t)((ks * LY::KV_TILE + (s >> 2) * EXT_BN * 128 + (s & 3) * 32) >> 4),
                                IDESC_S, s > 0 ? 1u : 0u);
                umma_commit(bar(LY::BAR_S + t));
            };
            auto issue_pv = [&](int t, int vs, int j, int h) {   // keys 64h .. 64h+63 of the tile
#pragma unroll
                for (int s = h * (EXT_BN / 32); s < (h + 1) * (EXT_BN / 32); ++s)
                    umma_f16_ts(tmem + LY::COL_O0 + t * D, tmem + t * EXT_BN + s * 8,
                                vd0 + (uint64_t)((vs * LY::KV_TILE + s * 16 * 128) >> 4), IDESC_PV,
                                (j > 0 || s > 0) ? 1u : 0u);
            };
            // The copies were made by the loaders' generic-proxy cp.async (and TMA) and are
            // acquired through the full barriers; a proxy fence orders them before the tensor
            // core's (async-proxy) reads.
            int gt = 0, ic = 0;               // K/V tiles and items consumed so far
            int sc0 = 0, sc1 = 0;             // score steps of Q tile 0 / 1 so far (barrier phases)
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int item = take_item_thread(k);
                if (item < 0) break;
                const ExtItem it = ext_item(p, item);
                if (!it.valid) continue;
                const int nt = it.ntiles, nkv = it.nkv;
                ok = mbar_wait(bar(LY::BAR_Q), ic & 1, abort_flag, p.status) &&
                     mbar_wait(bar(LY::BAR_KF + gt % NK), (gt / NK) & 1, abort_flag, p.status);
                ic += 1;
                if (!ok) break;
                fence_proxy_async_smem();
                tc_fence_after();
                for (int t = 0; t < nt; ++t) {
                    issue_s(t, gt % NK);
                    if (nkv == 1) umma_commit(bar(LY::BAR_QE + t));   // Q_t read by this item's last S
                }
                umma_commit(bar(LY::BAR_KE + gt % NK));
                for (int j = 0; ok && j < nkv; ++j) {
                    const int u = gt + j;
                    const int vs = u % NV;
                    if (!mbar_wait(bar(LY::BAR_VF + vs), (u / NV) & 1, abort_flag, p.status)) { ok = false; break; }
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const bool more = j + 1 < nkv;
                    const int ks = (u + 1) % NK;
                    for (int t = 0; t < nt; ++t) {
                        const int ph = ((t == 0 ? sc0 : sc1) + j) & 1;
                        // P arrives in two halves: PV over keys 0-63 runs while the softmax warps
                        // still compute keys 64-127
                        if (!mbar_wait(bar(LY::BAR_P + t), ph, abort_flag, p.status)) { ok = false; break; }
                        tc_fence_after();
                        issue_pv(t, vs, j, 0);
                        if (!mbar_wait(bar(LY::BAR_P + 2 + t), ph, abort_flag, p.status)) { ok = false; break; }
                        tc_fence_after();
                        issue_pv(t, vs, j, 1);
                        if (t == nt - 1) umma_commit(bar(LY::BAR_VE + vs));   // V(u) read by every tile
                        if (more) {
                            if (t == 0) {
                                if (!mbar_wait(bar(LY::BAR_KF + ks), ((u + 1) / NK) & 1, abort_flag, p.status)) {
                                    ok = false;
                                    break;
                                }
                                fence_proxy_async_smem();
                                tc_fence_after();
                            }
                            issue_s(t, ks);
                            if (j + 2 == nkv) umma_commit(bar(LY::BAR_QE + t));   // the item's last S_t
                        } else {
                            umma_commit(bar(LY::BAR_OR + t));   // O_t of this item complete
                        }
                    }
                    if (!ok) break;
                    if (more) umma_commit(bar(LY::BAR_KE + ks));
                }
                sc0 += nkv;
                sc1 += nt > 1 ? nkv : 0;
                gt += nkv;
            }
            umma_commit(bar(LY::BAR_DONE));
        }
        __syncwarp();
    }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        regs_increase<EXT_REGS_SOFTMAX>();
        const int t = wg - 1;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + t * EXT_BN;   // scores, then P over them
        const uint32_t o_addr = tmem + lane_base + LY::COL_O0 + t * D;
        const float sl = p.scale_log2;
        int sc = 0, oc = 0;                   // score steps and items of this Q tile so far
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = take_item_warp(k);
            if (item < 0) break;
            int pos, nkv;
            {
                // only what the score loop needs stays live through it; the epilogue decodes
                // the item again
                const ExtItem it = ext_item(p, item);
                if (!it.valid || t >= it.ntiles) continue;
                const int Rc = min(it.row0 + t * 128 + r, it.rows_total - 1);
                pos = p.shared_mode ? it.kv_end - 1 : it.P_b + Rc / G;   // attends keys 0..pos
                nkv = it.nkv;
            }
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < nkv; ++j) {
                if (!warp_wait(bar(LY::BAR_S + t), (sc + j) & 1, abort_flag, p.status)) { ok = false; break; }
                tc_fence_after();
                const int lim = pos - j * EXT_BN;   // columns past lim are masked
                if (__any_sync(0xffffffffu, lim < EXT_BN - 1)) {
                    // the diagonal tiles only: mask in TMEM, 32 columns at a time (rolled, to
                    // keep the loop's code small).  The whole warp enters (tcgen05.ld/st are
                    // warp-collective); a lane whose row sees the whole tile masks nothing.
#pragma unroll 1
                    for (int c0 = 0; c0 < EXT_BN; c0 += 32) {
                        float v[32];
                        tmem_ld32(s_addr + c0, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (c0 + e > lim) v[e] = -INFINITY;
                        tmem_st32(s_addr + c0, v);
                    }
                    tmem_wait_st();
                }
                float s[EXT_BN];
#pragma unroll
                for (int c = 0; c < EXT_BN; c += 32) tmem_ld32(s_addr + c, s + c);
                tmem_wait_ld();
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
                for (int c = 8; c + 16 <= EXT_BN; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[EXT_BN - 8 + i]);
                float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                mx *= sl;
                float m_new = m_ref;
                if (m_ref == -INFINITY || mx > m_ref + EXT_RESCALE_THRESHOLD) m_new = fmaxf(m_ref, mx);
                const float alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - m_new);
                const bool rescale = j > 0 && __any_sync(0xffffffffu, m_new != m_ref);
                l *= alpha;
                m_ref = m_new;
                const uint64_t sl2 = f2_pack(sl, sl), nm2 = f2_pack(-m_new, -m_new);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
                // P in two halves of 64 keys (32 columns), each published as soon as it is
                // stored, so that the tensor core starts PV on the first half
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[EXT_BN / 4];
#pragma unroll
                    for (int cc = 0; cc < EXT_BN / 2; cc += 2) {
                        const int c = h * (EXT_BN / 2) + cc;
                        const uint64_t x2 = f2_fma(f2_pack(s[c], s[c + 1]), sl2, nm2);
                        float x0, x1;
                        f2_unpack(x2, x0, x1);
                        const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
                        acc2[(c >> 1) & 3] = f2_add(acc2[(c >> 1) & 3], f2_pack(e0, e1));
                        pk[cc >> 1] = pack_bf16x2(e0, e1);
                    }
                    tmem_st32u(s_addr + h * 32, pk);
                    if (h == 0 && rescale) {
                        // PV_t(j-1) has completed (S_t(j) was issued after it and is complete),
                        // and PV_t(j) waits for the arrival below.  Rare: rolled.
#pragma unroll 1
                        for (int cc = 0; cc < D; cc += 32) {
                            float ov[32];
                            tmem_ld32(o_addr + cc, ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) ov[e] *= alpha;
                            tmem_st32(o_addr + cc, ov);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(LY::BAR_P + 2 * h + t));
                }
                const uint64_t a01 = f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3]));
                float ra, rb;
                f2_unpack(a01, ra, rb);
                l += ra + rb;
            }
            if (!ok) break;
            sc += nkv;
            const ExtItem it = ext_item(p, item);
            const int R = it.row0 + t * 128 + r;
            const bool valid = R < it.rows_total;
            const int Rc = min(R, it.rows_total - 1);
            const int tok = Rc / G;
            // The item's O_t is complete once its last PV has: the epilogue reads it while the
            // tensor core already works on the next item's scores; the next item's first PV
            // (which overwrites O_t) waits for P that this warpgroup publishes after the reads.
            if (!warp_wait(bar(LY::BAR_OR + t), oc & 1, abort_flag, p.status)) { ok = false; break; }
            oc += 1;
            tc_fence_after();
            const float inv = 1.f / l;
            if (p.shared_mode) {
                // fp32 normalised partial and log2-domain lse for the merge
                const int64_t row_item = (int64_t)p.grp_rows[it.m0 + tok] * p.hq + it.g * G + Rc % G;
                const int64_t slot = row_item * p.part_per + p.part_base + it.x % p.n_chunks;
                float* prow = p.part_o + slot * D;
#pragma unroll
                for (int cc = 0; cc < D; cc += 32) {
                    float ov[32];
                    tmem_ld32(o_addr + cc, ov);
                    tmem_wait_ld();
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(prow + cc + e) =
                                make_float4(ov[e] * inv, ov[e + 1] * inv, ov[e + 2] * inv, ov[e + 3] * inv);
                    }
                }
                if (valid) p.part_lse[slot] = m_ref + log2f(l);
            } else {
                // each thread writes its own normalised bf16 row (16-byte stores)
                __nv_bfloat16* orow = p.out + ((it.qo0 + tok) * p.hq + it.g * G + Rc % G) * D;
#pragma unroll
                for (int cc = 0; cc < D; cc += 32) {
                    float ov[32];
                    tmem_ld32(o_addr + cc, ov);
                    tmem_wait_ld();
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(ov[e + 0] * inv, ov[e + 1] * inv);
                            v.y = pack_bf16x2(ov[e + 2] * inv, ov[e + 3] * inv);
                            v.z = pack_bf16x2(ov[e + 4] * inv, ov[e + 5] * inv);
                            v.w = pack_bf16x2(ov[e + 6] * inv, ov[e + 7] * inv);
                            *reinterpret_cast<uint4*>(orow + cc + e) = v;
                        }
                    }
                }
                if (valid && p.lse) p.lse[(it.qo0 + tok) * p.hq + it.g * G + Rc % G] = (m_ref + log2f(l)) * EXT_LN2;
            }
            tc_fence_before();
        }
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    // The last CTA out resets the work counters for the next launch that uses them (launches
    // on one stream run one after another; every fetch of this CTA precedes its count).
    if (p.work && threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&p.work[1], 1u) == gridDim.x - 1) {
            atomicExch(&p.work[0], 0u);
            atomicExch(&p.work[1], 0u);
        }
    }
    if (warp == EXT_MMA_WARP) {
        tc_fence_after();
        // Every MMA this CTA issued has completed before TMEM is released; this wait does
        // not stop on the abort flag (only on its own time bound).
        volatile int no_abort = 0;
        warp_wait(bar(LY::BAR_DONE), 0, &no_abort, p.status, 500000000ull);
        tmem_dealloc(tmem, LY::TMEM_COLS);
    }
}

// The current device must be an sm_103 (GB300): checked once per device (a device that fails
// the check is checked again on the next call and fails again).
static int check_device() {
    static PerDeviceOnce checked;
    return per_device_once(checked, [] {
        int dev = 0, major = 0, minor = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            set_error("prefix_extend_attention: cannot query the device");
            return (int)RX_ECUDA;
        }
        if (major != 10 || minor != 3) {
            set_error("prefix_extend_attention: the tcgen05 kernel needs an sm_103 (GB300) device");
            return (int)RX_EDEVICE;
        }
        return (int)RX_OK;
    });
}

// cuTensorMapEncodeTiled from the driver, resolved once through the runtime (no -lcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Tensor map of a bf16 [rows][hq][D] buffer for the extend kernel's 128-row tiles: box
// 64 columns x G heads x 128/G tokens (a tile of packed rows, head fastest), 128-byte swizzle
// (the layout tcgen05 reads).  `rows` is the token extent of the map.  Returns false where the
// shape or address does not allow it (the kernel then gathers and stores row by row).
static bool rows_tensor_map(CUtensorMap* m, const void* ptr, int hq, int D, int G, int64_t rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || G <= 0 || 128 % G != 0 || (D != 64 && D != 128) || ((uintptr_t)ptr & 15u) != 0 || rows <= 0 ||
        rows > INT32_MAX)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hq, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hq * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    const cuuint32_t elem[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Streaming multiprocessors of the current device (one persistent CTA each), read once per device.
static int sm_count() {
    static PerDeviceOnce once;
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    per_device_once(once, [&] {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return (int)RX_ECUDA;
        counts[dev] = n;
        return (int)RX_OK;
    });
    return counts[dev];
}

// Work counters of the persistent grid, a pair per stream (launches on one stream run one after
// another and each launch's last CTA leaves its pair at zero; launches on different streams may
// overlap, so each stream has its own pair).  Zero when the module loads.
constexpr int EXT_WORK_SLOTS = 256;
__device__ unsigned int g_ext_work[EXT_WORK_SLOTS][2];

// The counter pair of `stream` on the current device, or null when every pair is taken (the
// kernel then walks its items round-robin).  The array's address is looked up on every call (a
// host-side lookup in the current context), so a context created after cudaDeviceReset, which
// loads the module at a new address with the counters at zero again, gets its own.
static unsigned int* work_counters(cudaStream_t stream) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> slot_of;   // (device, stream) -> pair
    static int used[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    void* base = nullptr;
    if (cudaGetSymbolAddress(&base, g_ext_work) != cudaSuccess || !base) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    const uint64_t key = ((uint64_t)dev << 56) ^ (uint64_t)(uintptr_t)stream;
    auto it = slot_of.find(key);
    if (it == slot_of.end()) {
        if (used[dev] >= EXT_WORK_SLOTS) return nullptr;
        it = slot_of.emplace(key, used[dev]++).first;
    }
    return (unsigned int*)base + 2 * it->second;
}

// Launches the kernel over the tiles x hkv x gz grid of work items as a persistent grid: one
// CTA per SM (at most one per item), taking the items in order from the stream's work counter.
template <int D>
static int launch_extend_tc(ExtendParams p, int tiles, cudaStream_t stream, int gz) {
    static PerDeviceOnce attr;
    const int smem = ExtLayout<D>::ALLOC;
    const int rc = per_device_once(attr, [&] {
        const cudaError_t e = cudaFuncSetAttribute(extend_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            set_error("prefix_extend_attention: cannot set shared memory size: %s", cudaGetErrorString(e));
            return (int)RX_ECUDA;
        }
        // The warpgroups re-split the registers the block is launched with (setmaxnreg); the
        // shares must add up to no more than that, or the increasing warps would wait forever.
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, extend_tc_kernel<D>) != cudaSuccess ||
            (int64_t)fa.numRegs * EXT_THREADS < 2 * 128 * (int64_t)EXT_REGS_OTHER + 2 * 128 * (int64_t)EXT_REGS_SOFTMAX) {
            set_error("prefix_extend_attention: kernel built with %d registers per thread; the register split needs %d",
                      fa.numRegs, (int)((2 * 128 * EXT_REGS_OTHER + 2 * 128 * EXT_REGS_SOFTMAX) / EXT_THREADS));
            return (int)RX_ECUDA;
        }
        return (int)RX_OK;
    });
    if (rc != RX_OK) return rc;
    const int64_t items = (int64_t)tiles * p.hkv * gz;
    if (items <= 0) return RX_OK;
    if (items >= (1ll << 31)) {
        set_error("prefix_extend_attention: too many work items (%lld)", (long long)items);
        return RX_EINVAL;
    }
    const int sms = sm_count();
    if (sms <= 0) {
        set_error("prefix_extend_attention: cannot read the device's SM count");
        return RX_ECUDA;
    }
    p.grid_x = tiles;
    p.n_items = (int32_t)items;
    // the counter only where a CTA walks several items: with at most one item per CTA (the
    // decode's shared-prefix part, launched beside the private part) each CTA takes its own
    p.work = items > sms ? work_counters(stream) : nullptr;
    const unsigned ctas = (unsigned)std::min<int64_t>(items, sms);
    extend_tc_kernel<D><<<ctas, EXT_THREADS, smem, stream>>>(p);
    return RX_OK;
}

// ---------------------------------------------------------------------------------------
// Grouped extend (requests sharing a cached prefix): the shared run is processed once for
// all members' stacked new rows on the tcgen05 kernel (partials per key chunk); each
// request's own tail (its private cached tokens and its new tokens, causally) on CUDA
// cores, merged exactly with the shared chunks:
//   M = max_s lse_s, o = sum_s 2^(lse_s-M) o_s / sum_s 2^(lse_s-M).
struct GroupedExtendWs {
    float* part_o;        // [T * hq][per][D]
    float* part_lse;      // [T * hq][per] (log2 domain)
    int32_t* row_indptr;  // [num_groups + 1]
    int32_t* rows;        // [T]
    int32_t* src;         // [num_groups]
    int32_t* shared_of;   // [batch] shared tokens of the request's group (0 outside groups)
    int32_t per;          // 1 (private) + shared chunks
};

// One block of 1024 threads: per-request shared lengths, the groups' row lists (members' new
// tokens, in member order) and source slot-table rows.  Members are processed 1024 at a time;
// each thread takes one member, a block-wide scan places its rows.
__global__ void __launch_bounds__(1024) grouped_prep_kernel(int32_t batch, const int64_t* qo_indptr, int32_t num_groups,
                                                           const int32_t* grp_indptr, const int32_t* grp_members,
                                                           const int32_t* grp_len, GroupedExtendWs ws, int32_t* status) {
    __shared__ int32_t scan[1024];
    __shared__ int32_t carry;
    for (int b = threadIdx.x; b < batch; b += blockDim.x) ws.shared_of[b] = 0;
    for (int gid = threadIdx.x; gid < num_groups; gid += blockDim.x)
        ws.src[gid] = (grp_indptr[gid + 1] > grp_indptr[gid]) ? grp_members[grp_indptr[gid]] : 0;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int M = grp_indptr[num_groups];
    for (int base = 0; base < M; base += 1024) {
        const int i = base + threadIdx.x;
        int b = -1, gid = 0, n = 0;
        int64_t q0 = 0;
        if (i < M) {
            b = grp_members[i];
            int lo = 0, hi = num_groups - 1;           // group of member i
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (grp_indptr[mid] <= i) lo = mid; else hi = mid - 1;
            }
            gid = lo;
            if (b >= 0 && b < batch) {
                q0 = qo_indptr[b];
                n = (int)(qo_indptr[b + 1] - q0);
            } else {
                report(status, RX_DEV_BAD_LENGTH);
                b = -1;
            }
        }
        scan[threadIdx.x] = n;
        __syncthreads();
        for (int off = 1; off < 1024; off <<= 1) {     // inclusive scan
            const int v = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
            __syncthreads();
            scan[threadIdx.x] += v;
            __syncthreads();
        }
        const int start = carry + scan[threadIdx.x] - n;
        if (i < M) {
            if (b >= 0) {
                ws.shared_of[b] = grp_len[gid];
                for (int t = 0; t < n; ++t) ws.rows[start + t] = (int32_t)(q0 + t);
            }
            if (i == grp_indptr[gid]) ws.row_indptr[gid] = start;   // first member of its group
        }
        __syncthreads();
        if (threadIdx.x == 1023) carry = start + n;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        ws.row_indptr[num_groups] = carry;
        for (int gid = num_groups - 1; gid >= 0; --gid)             // empty groups: empty row range
            if (grp_indptr[gid + 1] == grp_indptr[gid]) ws.row_indptr[gid] = ws.row_indptr[gid + 1];
    }
}

// Private part and merge: one warp per (new row, query head) attends keys
// [shared_of[b], P_b + i] of its own request on CUDA cores (its private cached tokens and its
// new tokens, causally), then merges that softmax part with the group's shared chunks.
template <int D>
__global__ void __launch_bounds__(128) grouped_private_merge_kernel(ExtendParams p, GroupedExtendWs ws,
                                                                    int64_t total_rows, int32_t chunk) {
    constexpr int E = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * 4 + warp;
    if (item >= total_rows * p.hq) return;
    const int64_t row = item / p.hq;
    if (row >= p.qo_indptr[p.batch]) return;
    const int h = (int)(item - row * p.hq);
    const int g = h / p.group;
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.qo_indptr[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int64_t i = row - p.qo_indptr[b];
    const int64_t n = p.qo_indptr[b + 1] - p.qo_indptr[b];
    const int64_t P = p.prefix_lens[b];
    if (n > p.max_qo_len || P < 0 || P + n > p.stride) {
        if (lane == 0 && h == 0 && i == 0) report(p.status, RX_DEV_BAD_LENGTH);
        return;
    }
    const int32_t shared = ws.shared_of[b];
    const int64_t pos = P + i;
    const __nv_bfloat16* qr = p.q + item * D;
    float qv[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        qv[e] = __bfloat162float(qr[lane + 32 * e]) * p.scale_log2;
        acc[e] = 0.f;
    }
    const int32_t* slots = p.r2t + (int64_t)b * p.stride;
    float m = -INFINITY, l = 0.f;
    for (int64_t j = shared; j <= pos; ++j) {
        const int32_t sl = slots[j];
        if (sl < 0 || sl >= p.num_slots) {
            if (lane == 0) report(p.status, RX_DEV_BAD_SLOT);
            continue;
        }
        const __nv_bfloat16* kr = p.k_pool + ((int64_t)sl * p.hkv + g) * D;
        const __nv_bfloat16* vr = p.v_pool + ((int64_t)sl * p.hkv + g) * D;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot += qv[e] * __bfloat162float(kr[lane + 32 * e]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float mn = fmaxf(m, dot);
        const float corr = exp2f(m - mn), w = exp2f(dot - mn);
        l = l * corr + w;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = acc[e] * corr + w * __bfloat162float(vr[lane + 32 * e]);
        m = mn;
    }
    // merge: private part (m, l, acc unnormalised) with the shared chunks (normalised, lse)
    const int nsh = (shared + chunk - 1) / chunk;
    const float* pl = ws.part_lse + item * ws.per;
    const float* po = ws.part_o + item * ws.per * D;
    const float lse_priv = m + log2f(l);              // -inf when the range was empty
    float M = lse_priv;
    for (int c = 0; c < nsh; ++c) M = fmaxf(M, pl[1 + c]);
    const float wp = (l > 0.f) ? exp2f(lse_priv - M) : 0.f;
    float W = wp, out[E];
#pragma unroll
    for (int e = 0; e < E; ++e) out[e] = (l > 0.f) ? wp * acc[e] / l : 0.f;
    for (int c = 0; c < nsh; ++c) {
        const float w = exp2f(pl[1 + c] - M);
        W += w;
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] += w * po[(int64_t)(1 + c) * D + lane + 32 * e];
    }
    __nv_bfloat16* orow = p.out + item * D;
#pragma unroll
    for (int e = 0; e < E; ++e) orow[lane + 32 * e] = __float2bfloat16_rn(out[e] / W);
    if (p.lse && lane == 0) p.lse[item] = (M + log2f(W)) * EXT_LN2;
}

static int grouped_chunk(int32_t max_group_len, int64_t row_tiles_x_heads) {
    // enough shared-part CTAs to cover the SMs, chunks of at least 128 keys
    int chunk = max_group_len;
    while (chunk > 128 && row_tiles_x_heads * ((max_group_len + chunk - 1) / chunk) < 152) chunk = (chunk + 1) / 2;
    return ((chunk + EXT_BN - 1) / EXT_BN) * EXT_BN;
}

struct GroupedLayout {
    int chunk, n_chunks, per;
    size_t o_bytes, lse_bytes, idx_bytes, total;
};

static GroupedLayout grouped_layout(const rx_attn_desc* d, int32_t batch, int64_t total_rows,
                                    const rx_shared_groups* grp) {
    GroupedLayout L{};
    const int G = d->hq / d->hkv;
    const int64_t row_tiles = ((int64_t)grp->max_group_rows * G + 255) / 256;
    L.chunk = grouped_chunk(grp->max_group_len, row_tiles * d->hkv);
    L.n_chunks = (grp->max_group_len + L.chunk - 1) / L.chunk;
    L.per = 1 + L.n_chunks;
    L.o_bytes = (size_t)total_rows * d->hq * L.per * d->head_dim * sizeof(float);
    L.lse_bytes = (size_t)total_rows * d->hq * L.per * sizeof(float);
    L.idx_bytes = ((size_t)(grp->num_groups + 1) + (size_t)total_rows + (size_t)grp->num_groups + (size_t)batch) *
                  sizeof(int32_t);
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    L.total = up(L.o_bytes) + up(L.lse_bytes) + up(L.idx_bytes);
    return L;
}

int launch_shared_prefix_tc(const SharedTcParams& sp, cudaStream_t stream) {
    const int dc = check_device();
    if (dc != RX_OK) return dc;
    ExtendParams p{};
    p.q = (const __nv_bfloat16*)sp.q;
    p.r2t = sp.r2t;
    p.stride = sp.stride;
    p.k_pool = (const __nv_bfloat16*)sp.k_pool;
    p.v_pool = (const __nv_bfloat16*)sp.v_pool;
    p.num_slots = sp.num_slots;
    p.batch = sp.batch;
    p.hq = sp.hq;
    p.hkv = sp.hkv;
    p.group = sp.hq / sp.hkv;
    p.scale_log2 = sp.scale * EXT_LOG2E;
    p.status = sp.status;
    p.shared_mode = 1;
    p.grp_row_indptr = sp.grp_row_indptr;
    p.grp_rows = sp.grp_rows;
    p.grp_src = sp.grp_src;
    p.grp_len = sp.grp_len;
    p.chunk = sp.chunk;
    p.n_chunks = sp.n_chunks;
    p.part_o = sp.part_o;
    p.part_lse = sp.part_lse;
    p.part_per = sp.part_per;
    p.part_base = sp.part_base;
    const int64_t row_tiles = ((int64_t)sp.max_group_rows * p.group + 255) / 256;
    const int64_t gx = row_tiles * sp.n_chunks;
    if (gx >= (1ll << 31) || sp.num_groups >= 65536) {
        set_error("decode_attention: shared-prefix grid too large");
        return RX_EINVAL;
    }
    const int rc = sp.head_dim == 128 ? launch_extend_tc<128>(p, (int)gx, stream, sp.num_groups)
                                      : launch_extend_tc<64>(p, (int)gx, stream, sp.num_groups);
    if (rc != RX_OK) return rc;
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("decode_attention: shared-prefix launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

}  // namespace rx

using namespace rx;

extern "C" size_t extend_workspace_bytes(const rx_attn_desc* desc, int32_t batch, int32_t max_qo_len,
                                         const rx_shared_groups* groups) {
    if (!desc || batch < 0 || max_qo_len < 0 || desc->hkv <= 0 || desc->hq % desc->hkv != 0) return 0;
    if (!groups || groups->num_groups <= 0) return 0;
    return grouped_layout(desc, batch, (int64_t)batch * max_qo_len, groups).total;
}

static int grouped_extend(const rx_attn_desc* desc, const ExtendParams& p, const rx_shared_groups* groups,
                          void* d_workspace, size_t ws_bytes, cudaStream_t stream) {
    RX_REQUIRE(groups->d_group_indptr && groups->d_group_members && groups->d_group_len &&
                   groups->max_group_rows >= 1 && groups->max_group_len >= 1,
               "prefix_extend_attention: incomplete shared groups");
    const int64_t rows_bound = (int64_t)p.batch * p.max_qo_len;
    const GroupedLayout L = grouped_layout(desc, p.batch, rows_bound, groups);
    RX_REQUIRE(d_workspace && ws_bytes >= L.total && ((uintptr_t)d_workspace & 255) == 0,
               "prefix_extend_attention: grouped path needs a 256-byte aligned workspace of %zu bytes (got %zu)",
               L.total, ws_bytes);
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    unsigned char* w = (unsigned char*)d_workspace;
    GroupedExtendWs ws{};
    ws.part_o = (float*)w;
    ws.part_lse = (float*)(w + up(L.o_bytes));
    int32_t* idx = (int32_t*)(w + up(L.o_bytes) + up(L.lse_bytes));
    ws.row_indptr = idx;
    ws.rows = idx + groups->num_groups + 1;
    ws.src = ws.rows + rows_bound;
    ws.shared_of = ws.src + groups->num_groups;
    ws.per = L.per;
    grouped_prep_kernel<<<1, 1024, 0, stream>>>(p.batch, p.qo_indptr, groups->num_groups, groups->d_group_indptr,
                                                 groups->d_group_members, groups->d_group_len, ws, p.status);
    SharedTcParams sp{};
    sp.q = p.q;
    sp.r2t = p.r2t;
    sp.stride = p.stride;
    sp.k_pool = p.k_pool;
    sp.v_pool = p.v_pool;
    sp.num_slots = p.num_slots;
    sp.batch = p.batch;
    sp.hq = p.hq;
    sp.hkv = p.hkv;
    sp.head_dim = desc->head_dim;
    sp.scale = desc->scale;
    sp.status = p.status;
    sp.num_groups = groups->num_groups;
    sp.max_group_rows = groups->max_group_rows;
    sp.grp_row_indptr = ws.row_indptr;
    sp.grp_rows = ws.rows;
    sp.grp_src = ws.src;
    sp.grp_len = groups->d_group_len;
    sp.chunk = L.chunk;
    sp.n_chunks = L.n_chunks;
    sp.part_o = ws.part_o;
    sp.part_lse = ws.part_lse;
    sp.part_per = L.per;
    sp.part_base = 1;
    int rc = launch_shared_prefix_tc(sp, stream);
    if (rc != RX_OK) return rc;
    const int64_t items = rows_bound * p.hq;
    const unsigned blocks = (unsigned)((items + 3) / 4);
    if (desc->head_dim == 128)
        grouped_private_merge_kernel<128><<<blocks, 128, 0, stream>>>(p, ws, rows_bound, L.chunk);
    else
        grouped_private_merge_kernel<64><<<blocks, 128, 0, stream>>>(p, ws, rows_bound, L.chunk);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("prefix_extend_attention: grouped launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

extern "C" int prefix_extend_attention(const rx_attn_desc* desc, int32_t batch, const void* d_q,
                                       const int64_t* d_qo_indptr, const int32_t* d_prefix_lens,
                                       const int32_t* d_req_to_token, int64_t r2t_stride, const void* d_k_pool,
                                       const void* d_v_pool, void* d_out, float* d_lse, int32_t max_qo_len,
                                       const rx_shared_groups* groups, void* d_workspace, size_t ws_bytes,
                                       int32_t* d_status, void* stream_) {
    RX_TRACE("prefix_extend_attention");
    RX_REQUIRE(desc && batch >= 0 && max_qo_len >= 0 && r2t_stride >= 0, "prefix_extend_attention: bad arguments");
    RX_REQUIRE(desc->hq > 0 && desc->hkv > 0 && desc->hq % desc->hkv == 0,
               "prefix_extend_attention: bad head counts");
    RX_REQUIRE(desc->head_dim == 64 || desc->head_dim == 128, "prefix_extend_attention: head_dim must be 64 or 128");
    if (batch == 0 || max_qo_len == 0) return RX_OK;
    RX_REQUIRE(d_q && d_qo_indptr && d_prefix_lens && d_req_to_token && d_k_pool && d_v_pool && d_out,
               "prefix_extend_attention: null device pointer");
    cudaStream_t stream = (cudaStream_t)stream_;
    const int group = desc->hq / desc->hkv;
    if (desc->dtype == RX_F32) {
        // fp32 keeps fp32 arithmetic on CUDA cores; rows are sized by the host bound.
        SimtParams sp{};
        sp.batch = batch;
        sp.hq = desc->hq;
        sp.hkv = desc->hkv;
        sp.total_rows = -1;
        sp.q = d_q;
        sp.qo_indptr = d_qo_indptr;
        sp.prefix_lens = d_prefix_lens;
        sp.r2t = d_req_to_token;
        sp.stride = r2t_stride;
        sp.k_pool = d_k_pool;
        sp.v_pool = d_v_pool;
        sp.num_slots = desc->num_slots;
        sp.out = d_out;
        sp.lse = d_lse;
        sp.scale = desc->scale;
        sp.max_len = max_qo_len;
        sp.status = d_status;
        // Rows are bounded by batch * max_qo_len; rows past qo_indptr[batch] exit at once.
        sp.total_rows = (int64_t)batch * max_qo_len;
        return launch_attn_simt(sp, desc->dtype, desc->head_dim, stream);
    }
    RX_REQUIRE(desc->dtype == RX_BF16, "prefix_extend_attention: unknown dtype %d", desc->dtype);
    const int dc = check_device();
    if (dc != RX_OK) return dc;
    ExtendParams p{};
    p.q = (const __nv_bfloat16*)d_q;
    p.qo_indptr = d_qo_indptr;
    p.prefix_lens = d_prefix_lens;
    p.r2t = d_req_to_token;
    p.stride = r2t_stride;
    p.k_pool = (const __nv_bfloat16*)d_k_pool;
    p.v_pool = (const __nv_bfloat16*)d_v_pool;
    p.num_slots = desc->num_slots;
    p.out = (__nv_bfloat16*)d_out;
    p.lse = d_lse;
    p.batch = batch;
    p.hq = desc->hq;
    p.hkv = desc->hkv;
    p.group = group;
    p.scale_log2 = desc->scale * EXT_LOG2E;
    p.max_qo_len = max_qo_len;
    p.status = d_status;
    if (groups && groups->num_groups > 0) return grouped_extend(desc, p, groups, d_workspace, ws_bytes, stream);
    if ((int64_t)group * max_qo_len <= SMALL_EXT_MAX_ROWS && r2t_stride <= SMALL_EXT_MAX_KEYS) {
        // a handful of rows per (request, kv head) over at most 1024 keys: the decode-shaped
        // kernel (keys in M of mma.sync, the rows in N) in one chunk, final rows written directly
        SmallExtendArgs a{};
        a.q = d_q;
        a.qo_indptr = d_qo_indptr;
        a.prefix_lens = d_prefix_lens;
        a.r2t = d_req_to_token;
        a.stride = r2t_stride;
        a.k_pool = d_k_pool;
        a.v_pool = d_v_pool;
        a.num_slots = desc->num_slots;
        a.out = d_out;
        a.lse = d_lse;
        a.batch = batch;
        a.hq = desc->hq;
        a.hkv = desc->hkv;
        a.head_dim = desc->head_dim;
        a.max_qo_len = max_qo_len;
        a.scale = desc->scale;
        a.status = d_status;
        RX_REQUIRE(batch < 65536, "prefix_extend_attention: grid too large");
        return launch_extend_small(a, stream);
    }
    const int64_t tiles = ((int64_t)max_qo_len * group + 255) / 256;
    RX_REQUIRE(tiles < 65536 && batch < 65536, "prefix_extend_attention: grid too large");
    // The rows of q and out are located through qo_indptr, whose first entry need not be 0,
    // so the host knows no tighter bound than the 31-bit coordinate range: the maps never
    // clip, and the kernel addresses through them only full tiles of one request's rows
    // (the rows the row-by-row path would touch as well).
    const int64_t row_bound = INT32_MAX;
    p.q_map_ok = rows_tensor_map(&p.q_map, d_q, desc->hq, desc->head_dim, group, row_bound) ? 1 : 0;
    const int rc = desc->head_dim == 128 ? launch_extend_tc<128>(p, (int)tiles, stream, batch)
                                         : launch_extend_tc<64>(p, (int)tiles, stream, batch);
    if (rc != RX_OK) return rc;
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("prefix_extend_attention: launch failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}
