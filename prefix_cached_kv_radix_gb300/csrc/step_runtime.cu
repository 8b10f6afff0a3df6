// One-call launch of a planned step: the copy of the step's index arrays, kv_pool_write, the
// attention call and the host-side finish (insert, evict, unpin), so that a serving loop
// crosses the library boundary twice per step (rx_step_plan, rx_step_launch) instead of once
// per operation.  "SGLang: Efficient Execution of Structured Language Model Programs",
// RadixAttention: per request, match the cached prefix, compute only the new tokens against
// it, insert them, evict under memory pressure.
//
// The staging buffer a step was planned into is read by an asynchronous copy; each staging
// buffer has an event (recorded after its copy) that rx_stage_wait synchronises, so the next
// plan into the same buffer cannot overwrite it early.
//
// With host buffers the step's rows cross the host link inside the call, as a pipeline of
// request ranges: range c+1's rows are copied in (copy-in stream) while range c runs
// kv_pool_write and attention (the caller's stream) and range c-1's output is copied out
// (copy-out stream), so the transfers hide behind the kernels instead of adding to them.
// Ranges need no other synchronisation: a request's prefix slots were all written by earlier
// steps, and its own new K/V by its own range.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <chrono>
#include <mutex>
#include <thread>
#include <unordered_map>
#include <vector>

#include "radix_attn.h"
#include "rx_common.h"
#include "rx_kernels.h"

namespace rx {

// NVTX ranges of the ABI calls (only reached when tracing is on): NVTX's header-only dispatch
// forwards them to an attached profiler and ignores them otherwise.
void trace_push(const char* name) { nvtxRangePushA(name); }
void trace_pop() { nvtxRangePop(); }

}  // namespace rx

namespace {

std::mutex g_ev_mu;
struct StageInfo {
    cudaEvent_t ev = nullptr;         // recorded after the last reads of the staging buffer
    void* h_dev = nullptr;            // its device mapping (null: not mapped)
    bool mapped_known = false;
    // Small device-row steps: kv_pool_write is the staging buffer's only reader, and its last
    // block writes `seq` to flag_host (pinned, mapped; flag_dev on the device) when the launch
    // is done with the buffer, counting its blocks in ctr_dev (device memory on `dev`).  Then
    // no event is recorded, and waiting is reading host memory.
    uint32_t* flag_host = nullptr;
    uint32_t* flag_dev = nullptr;
    unsigned* ctr_dev = nullptr;
    int dev = -1;
    uint32_t seq = 0;
    int mode = 0;                     // the last launch's reads end at: 0 nothing, 1 ev, 2 flag == seq
};
std::unordered_map<const void*, StageInfo> g_stage_events;   // staging buffer -> its event and mapping

// The index arrays of a host-buffer step, read by the GPU straight from the pinned staging
// buffer (mapped into the device's address space) instead of by a copy engine, so that they
// never wait behind the bulk row copies queued on the engines.  16-byte vectors, four
// independent loads per thread in flight (reads across the host link are latency-bound).
__global__ void __launch_bounds__(256) stage_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n; i += stride) dst[i] = src[i];
}

// Copy streams and events of the host-buffer pipeline, per device (created on first use),
// and the input copies a rx_step_prefetch has started for the next rx_step_launch.
struct Pipe {
    cudaStream_t in = nullptr, out = nullptr;
    std::vector<cudaEvent_t> ev;      // start, end, then per range: in, done
    std::mutex use;                   // one step enqueues on a device's pipe at a time
    bool pending = false;             // copies started by rx_step_prefetch, not yet used
    const void* p_hq = nullptr;
    const void* p_dq = nullptr;
    int64_t p_T = 0;
    std::vector<int32_t> p_cut;       // the request ranges they were cut into
    // Release events of device input rows: recorded on the compute stream after the kernels of
    // the last host-buffer step that read the rows at d_q (the last four buffers).
    struct Release {
        const void* d_q = nullptr;
        cudaEvent_t ev = nullptr;
    };
    Release rel[4];
    int rel_next = 0;
    // The same for device staging buffers (d_stage) of device-row steps with overlap, whose
    // index-array copy runs on the copy-in stream; `staged` marks the copy's completion.
    Release srel[4];
    int srel_next = 0;
    cudaEvent_t staged = nullptr;
};

// The release event of `buf` in table r (n entries, round robin), created on first use.
cudaError_t release_slot(Pipe::Release* r, int n, int* next, const void* buf, cudaEvent_t* out) {
    for (int i = 0; i < n; ++i)
        if (r[i].ev && r[i].d_q == buf) {
            *out = r[i].ev;
            return cudaSuccess;
        }
    Pipe::Release& x = r[*next];
    *next = (*next + 1) % n;
    if (!x.ev) {
        const cudaError_t e = cudaEventCreateWithFlags(&x.ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    x.d_q = buf;
    *out = x.ev;
    return cudaSuccess;
}

cudaEvent_t release_of(const Pipe::Release* r, int n, const void* buf) {
    for (int i = 0; i < n; ++i)
        if (r[i].ev && r[i].d_q == buf) return r[i].ev;
    return nullptr;
}
std::mutex g_pipe_mu;
std::unordered_map<int, Pipe> g_pipes;

int pipe_for(int nev, Pipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        rx::set_error("rx_step_launch: cannot query the device");
        return RX_ECUDA;
    }
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    Pipe& p = g_pipes[dev];
    if (!p.in && (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
                  cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess)) {
        rx::set_error("rx_step_launch: cannot create the copy streams");
        return RX_ECUDA;
    }
    while ((int)p.ev.size() < nev) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            rx::set_error("rx_step_launch: cannot create an event");
            return RX_ECUDA;
        }
        p.ev.push_back(e);
    }
    *out = &p;
    return RX_OK;
}

// Row bytes of the step's tensors: q/out rows (hq heads) and k/v rows (hkv heads).
struct RowBytes {
    int64_t q, kv;
};
RowBytes row_bytes(const rx_attn_desc* d) {
    const int64_t elt = d->dtype == RX_F32 ? 4 : 2;
    return {(int64_t)d->hq * d->head_dim * elt, (int64_t)d->hkv * d->head_dim * elt};
}

// The pipeline's request ranges, cut at request boundaries of the row index qo (host, batch+1
// entries): `chunks` ranges of about equal token counts; or, for chunks = 0, one range per 64 MB
// moved (at most 4), with the last eighth of the last range's tokens (at least one request) cut
// off as a range of its own when there are several: the output copy of the step's last range is
// the one copy that no later kernel of the step hides, so it is kept short.
std::vector<int32_t> range_cuts(const rx_attn_desc* d, const int64_t* qo, int32_t B, int32_t chunks) {
    const int64_t T = qo[B] - qo[0];
    const RowBytes rb = row_bytes(d);
    int nc = chunks > 0 ? chunks : (int)std::min<int64_t>(4, std::max<int64_t>(1, (T * (2 * rb.q + 2 * rb.kv)) >> 26));
    nc = std::max(1, std::min<int>(nc, std::max(B, 1)));
    std::vector<int32_t> cut((size_t)nc + 1, 0);
    cut[(size_t)nc] = B;
    for (int c = 1; c < nc; ++c) {   // first request whose rows start at or after c/nc of the tokens
        const int64_t target = qo[0] + T * c / nc;
        cut[(size_t)c] = std::max((int32_t)(std::lower_bound(qo, qo + B, target) - qo), cut[(size_t)c - 1]);
    }
    if (chunks <= 0 && nc > 1) {
        const int32_t b0 = cut[(size_t)nc - 1];
        if (B - b0 >= 2) {             // the first request whose rows start in the last eighth
            const int64_t target = qo[B] - (qo[B] - qo[b0]) / 8;
            int32_t s = (int32_t)(std::lower_bound(qo + b0 + 1, qo + B, target) - qo);
            s = std::min(s, B - 1);
            cut.insert(cut.end() - 1, s);
        }
    }
    return cut;
}

// The input copies of ranges c_begin .. c_end-1: on `stream` itself for a single range, else
// on the copy-in stream, each range's completion recorded in its event.  `start`: the copy
// streams first wait for the work already on `stream` (the first copies of a step) -- with
// io->overlap, only for the kernels of the last step that read io->d_q, when it is tracked.
int copy_in(Pipe* pp, const rx_attn_desc* d, const rx_step_io* io, const int64_t* qo, const std::vector<int32_t>& cut,
            int c_begin, int c_end, bool start, cudaStream_t stream) {
    const RowBytes rb = row_bytes(d);
    const int nc = (int)cut.size() - 1;
    cudaStream_t s_in = nc > 1 ? pp->in : stream;
    cudaError_t e = cudaSuccess;
    if (nc > 1 && start) {
        cudaEvent_t w = io->overlap ? release_of(pp->rel, 4, io->d_q) : nullptr;
        if (!w) {
            w = pp->ev[0];
            e = cudaEventRecord(w, stream);
        }
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, w, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(pp->out, w, 0);
    }
    for (int c = c_begin; c < c_end && e == cudaSuccess; ++c) {
        const int64_t t0 = qo[cut[(size_t)c]], t1 = qo[cut[(size_t)c + 1]];
        if (t1 > t0) {
            e = cudaMemcpyAsync((char*)io->d_q + t0 * rb.q, (const char*)io->h_q + t0 * rb.q, (size_t)((t1 - t0) * rb.q),
                                cudaMemcpyHostToDevice, s_in);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync((char*)io->d_k_new + t0 * rb.kv, (const char*)io->h_k_new + t0 * rb.kv,
                                    (size_t)((t1 - t0) * rb.kv), cudaMemcpyHostToDevice, s_in);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync((char*)io->d_v_new + t0 * rb.kv, (const char*)io->h_v_new + t0 * rb.kv,
                                    (size_t)((t1 - t0) * rb.kv), cudaMemcpyHostToDevice, s_in);
        }
        if (e == cudaSuccess && nc > 1) e = cudaEventRecord(pp->ev[2 + 2 * c], s_in);
    }
    if (e != cudaSuccess) {
        rx::set_error("rx_step_launch: input copy failed: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

rx_shared_groups groups_of(const rx_step_layout* L, unsigned char* d_stage) {
    rx_shared_groups g{};
    g.num_groups = L->num_groups;
    g.max_group_size = L->max_group_size;
    g.d_group_indptr = (const int32_t*)(d_stage + L->off_grp_indptr);
    g.d_group_members = (const int32_t*)(d_stage + L->off_grp_members);
    g.d_group_len = (const int32_t*)(d_stage + L->off_grp_len);
    g.max_group_len = L->max_group_len;
    g.max_group_rows = L->max_group_rows;
    return g;
}

}  // namespace

using rx::set_error;

extern "C" size_t rx_step_workspace_bytes(const rx_attn_desc* desc, const rx_step_layout* L, int32_t decode) {
    if (!desc || !L) return 0;
    rx_shared_groups g{};
    const rx_shared_groups* gp = nullptr;
    if (L->num_groups > 0) {
        g = groups_of(L, nullptr);
        gp = &g;
    }
    return decode ? decode_workspace_bytes(desc, L->batch, L->max_kv_len, gp)
                  : extend_workspace_bytes(desc, L->batch, L->max_qo_len, gp);
}

// The staging buffer's completion flag and block counter on the current device, made on the
// buffer's first small device-row launch there (the counter is cleared on `stream`, ahead of
// that launch).  RX_OK when the buffer can use them on this device.
static int stage_flag(StageInfo* si, cudaStream_t stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RX_ECUDA;
    }
    std::lock_guard<std::mutex> lk(g_ev_mu);
    if (si->flag_host) return si->dev == dev ? RX_OK : RX_EINVAL;
    void* h = nullptr;
    void* d = nullptr;
    void* c = nullptr;
    if (cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess ||
        cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess || cudaMalloc(&c, 64) != cudaSuccess ||
        cudaMemsetAsync(c, 0, 64, stream) != cudaSuccess) {
        cudaGetLastError();
        if (c) cudaFree(c);
        if (h) cudaFreeHost(h);
        return RX_ECUDA;
    }
    si->flag_host = (uint32_t*)h;
    *si->flag_host = 0;
    si->flag_dev = (uint32_t*)d;
    si->ctr_dev = (unsigned*)c;
    si->dev = dev;
    si->seq = 0;
    return RX_OK;
}

// Wait until *flag == seq: first by reading it (the GPU is usually done by the time the host
// gets here), then with short sleeps while checking the context for a fault, for at most a
// minute.  The acquire load orders the caller's later writes to the staging buffer after it.
static int wait_stage_flag(const uint32_t* flag, uint32_t seq) {
    for (int i = 0; i < 4096; ++i)
        if (__atomic_load_n(flag, __ATOMIC_ACQUIRE) == seq) return RX_OK;
    const auto t0 = std::chrono::steady_clock::now();
    while (__atomic_load_n(flag, __ATOMIC_ACQUIRE) != seq) {
        const cudaError_t e = cudaStreamQuery(0);   // reports an earlier fault; does not wait
        if (e != cudaSuccess && e != cudaErrorNotReady) {
            set_error("rx_stage_wait: %s", cudaGetErrorString(e));
            return RX_ECUDA;
        }
        if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(60)) {
            set_error("rx_stage_wait: the staging buffer's last launch has not finished after 60 s");
            return RX_ECUDA;
        }
        std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
    return RX_OK;
}

extern "C" int rx_stage_wait(const void* h_stage) {
    RX_TRACE("rx_stage_wait");
    cudaEvent_t ev = nullptr;
    const uint32_t* flag = nullptr;
    uint32_t seq = 0;
    {
        std::lock_guard<std::mutex> lk(g_ev_mu);
        auto it = g_stage_events.find(h_stage);
        if (it != g_stage_events.end()) {
            if (it->second.mode == 1) ev = it->second.ev;
            if (it->second.mode == 2) {
                flag = it->second.flag_host;
                seq = it->second.seq;
            }
        }
    }
    if (flag) return wait_stage_flag(flag, seq);
    if (!ev) return RX_OK;
    const cudaError_t e = cudaEventSynchronize(ev);
    if (e != cudaSuccess) {
        set_error("rx_stage_wait: %s", cudaGetErrorString(e));
        return RX_ECUDA;
    }
    return RX_OK;
}

extern "C" int rx_step_launch(rx_radix* t, const rx_attn_desc* desc, const int32_t* tokens, const int64_t* tok_indptr,
                              const rx_node* last_nodes, void* h_stage, const rx_step_layout* L, const rx_step_io* io,
                              int64_t evict_tokens, int64_t* out_evicted, void* stream_) {
    RX_TRACE("rx_step_launch");
    RX_REQUIRE(t && desc && L && io && h_stage && tok_indptr, "rx_step_launch: bad arguments");
    const int32_t B = L->batch;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (B > 0 && L->total_new > 0) {
        RX_REQUIRE(io->d_stage && io->d_stage_bytes >= (size_t)L->bytes, "rx_step_launch: device staging of %zu bytes, %lld needed",
                   io->d_stage_bytes, (long long)L->bytes);
        RX_REQUIRE(io->d_r2t && io->r2t_elems >= (int64_t)B * L->stride, "rx_step_launch: slot table of %lld entries, %lld needed",
                   (long long)io->r2t_elems, (long long)B * L->stride);
        RX_REQUIRE(!io->decode || L->max_qo_len == 1, "rx_step_launch: decode needs exactly one new token per request");
        const size_t ws = rx_step_workspace_bytes(desc, L, io->decode);
        RX_REQUIRE(ws == 0 || (io->d_workspace && io->ws_bytes >= ws), "rx_step_launch: workspace of %zu bytes, %zu needed",
                   io->ws_bytes, ws);
        // the staging buffer's event and device mapping, looked up once per buffer
        cudaEvent_t ev = nullptr;
        void* h_map = nullptr;
        StageInfo* sinfo = nullptr;
        {
            std::lock_guard<std::mutex> lk(g_ev_mu);
            StageInfo& si = g_stage_events[h_stage];
            sinfo = &si;   // entries are never erased: the reference stays valid
            if (!si.ev && cudaEventCreateWithFlags(&si.ev, cudaEventDisableTiming) != cudaSuccess) {
                si.ev = nullptr;
                set_error("rx_step_launch: cannot create an event");
                return RX_ECUDA;
            }
            if (!si.mapped_known) {
                if (cudaHostGetDevicePointer(&si.h_dev, h_stage, 0) != cudaSuccess) {
                    cudaGetLastError();   // not mapped (pageable): clear the error, copy instead
                    si.h_dev = nullptr;
                }
                si.mapped_known = true;
            }
            ev = si.ev;
            h_map = si.h_dev;
        }
        unsigned char* ds = (unsigned char*)io->d_stage;
        const int32_t* prefix_slots = (const int32_t*)(ds + L->off_prefix_slots);
        const int64_t* prefix_indptr = (const int64_t*)(ds + L->off_prefix_indptr);
        const int32_t* new_slots = (const int32_t*)(ds + L->off_new_slots);
        const int64_t* qo_indptr = (const int64_t*)(ds + L->off_qo_indptr);
        const int32_t* prefix_lens = (const int32_t*)(ds + L->off_prefix_lens);
        const int32_t* kv_lens = (const int32_t*)(ds + L->off_kv_lens);
        rx_shared_groups g{};
        const rx_shared_groups* gp = nullptr;
        if (L->num_groups > 0) {
            g = groups_of(L, ds);
            gp = &g;
        }
        const bool host = io->h_q != nullptr;
        if (host)
            RX_REQUIRE(io->h_k_new && io->h_v_new && io->h_out, "rx_step_launch: host-buffer mode needs h_k_new, h_v_new, h_out");
        const RowBytes rb = row_bytes(desc);
        const int64_t* h_qo = (const int64_t*)((const unsigned char*)h_stage + L->off_qo_indptr);
        // the index arrays: read by a kernel through the mapping of the pinned staging buffer
        // when it has one -- in host-buffer mode (never behind the rows' copies) and for small
        // arrays (a copy-engine transfer costs more in fixed latency there) -- otherwise one
        // copy-engine transfer (about twice the kernel's rate over the host link)
        constexpr int64_t kSmallStage = 1 << 20;
        const bool by_kernel = host || L->bytes <= kSmallStage;
        void* h_dev = by_kernel ? h_map : nullptr;
        cudaError_t e = cudaSuccess;
        // device rows, small arrays: kv_pool_write reads the slot lists from the mapping itself
        // and copies the whole buffer for the attention kernels in the same launch (one launch
        // fewer); the event follows it
        bool fused_stage = false;
        // device rows with overlap: the copy runs on the copy-in stream, after the kernels that
        // last read this d_stage (when tracked; else after all work on `stream`), and `stream`
        // waits for it -- under the previous step's kernels when the caller alternates d_stage
        Pipe* sp = nullptr;
        std::unique_lock<std::mutex> stage_lock;
        if (!by_kernel && io->overlap) {
            int rc = pipe_for(2, &sp);
            if (rc != RX_OK) return rc;
            stage_lock = std::unique_lock<std::mutex>(sp->use);
            if (!sp->staged) e = cudaEventCreateWithFlags(&sp->staged, cudaEventDisableTiming);
            cudaEvent_t w = release_of(sp->srel, 4, io->d_stage);
            if (e == cudaSuccess && !w) {
                w = sp->ev[0];
                e = cudaEventRecord(w, stream);
            }
            if (e == cudaSuccess) e = cudaStreamWaitEvent(sp->in, w, 0);
            if (e == cudaSuccess) e = cudaMemcpyAsync(io->d_stage, h_stage, (size_t)L->bytes, cudaMemcpyHostToDevice, sp->in);
            if (e == cudaSuccess) e = cudaEventRecord(ev, sp->in);
            if (e == cudaSuccess) e = cudaEventRecord(sp->staged, sp->in);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, sp->staged, 0);
        } else if (h_dev && ((uintptr_t)h_dev & 15) == 0 && ((uintptr_t)io->d_stage & 15) == 0 && L->bytes % 16 == 0 &&
                   !host) {
            fused_stage = true;
        } else if (h_dev && ((uintptr_t)h_dev & 15) == 0 && ((uintptr_t)io->d_stage & 15) == 0 && L->bytes % 16 == 0) {
            const int64_t n = L->bytes / 16;
            const int blocks = (int)std::min<int64_t>(152 * 2, (n + 255) / 256);
            stage_copy_kernel<<<std::max(blocks, 1), 256, 0, stream>>>((const uint4*)h_dev, (uint4*)io->d_stage, n);
            e = cudaGetLastError();
            if (e == cudaSuccess) e = cudaEventRecord(ev, stream);
        } else {
            e = cudaMemcpyAsync(io->d_stage, h_stage, (size_t)L->bytes, cudaMemcpyHostToDevice, stream);
            if (e == cudaSuccess) e = cudaEventRecord(ev, stream);
        }
        if (e != cudaSuccess) {
            set_error("rx_step_launch: staging copy failed: %s", cudaGetErrorString(e));
            return RX_ECUDA;
        }
        if (!fused_stage) {   // the event just recorded marks the end of the buffer's reads
            std::lock_guard<std::mutex> lk(g_ev_mu);
            sinfo->mode = 1;
        }
        std::vector<int32_t> cut{0, B};
        Pipe* pp = nullptr;
        std::unique_lock<std::mutex> pipe_lock;
        if (host) {
            int rc = pipe_for(2, &pp);
            if (rc != RX_OK) return rc;
            pipe_lock = std::unique_lock<std::mutex>(pp->use);
            if (pp->pending && pp->p_hq == io->h_q && pp->p_dq == io->d_q) {
                // the first range is already on its way (rx_step_prefetch, same ranges cut from
                // n_new): the rest follow the index arrays
                RX_REQUIRE(pp->p_T == L->total_new && pp->p_cut.back() == B,
                           "rx_step_launch: the prefetched rows are not this step's (%lld rows, %lld prefetched)",
                           (long long)L->total_new, (long long)pp->p_T);
                cut = pp->p_cut;
                rc = copy_in(pp, desc, io, h_qo, cut, 1, (int)cut.size() - 1, false, stream);
            } else {
                cut = range_cuts(desc, h_qo, B, io->chunks);
                rc = pipe_for(2 + 2 * ((int)cut.size() - 1), &pp);
                if (rc == RX_OK) rc = copy_in(pp, desc, io, h_qo, cut, 0, (int)cut.size() - 1, true, stream);
            }
            if (rc != RX_OK) return rc;
            pp->pending = false;
        }
        const int nc = (int)cut.size() - 1;
        // shared-prefix groups span ranges: then one compute over all rows once every range is in
        const bool ranged = nc > 1 && gp == nullptr;
        if (nc > 1 && !ranged)
            for (int c = 0; c < nc && e == cudaSuccess; ++c) e = cudaStreamWaitEvent(stream, pp->ev[2 + 2 * c], 0);
        const int nk = ranged ? nc : 1;
        for (int c = 0; c < nk && e == cudaSuccess; ++c) {
            const int32_t b0 = ranged ? cut[(size_t)c] : 0, b1 = ranged ? cut[(size_t)c + 1] : B;
            if (b1 == b0) continue;
            if (ranged) e = cudaStreamWaitEvent(stream, pp->ev[2 + 2 * c], 0);
            if (e != cudaSuccess) break;
            const int64_t t0 = h_qo[b0], t1 = h_qo[b1];
            const int32_t nb = b1 - b0;
            int32_t* r2t_c = io->d_r2t + (int64_t)b0 * L->stride;
            int rc;
            if (fused_stage) {   // one range (device rows): the index arrays from the mapping
                const unsigned char* hm = (const unsigned char*)h_dev;
                // the launch's end is signalled in host memory when this buffer has a flag on
                // this device, else by the event
                const bool by_flag = stage_flag(sinfo, stream) == RX_OK;
                uint32_t seq = 0;
                if (by_flag) {
                    std::lock_guard<std::mutex> lk(g_ev_mu);
                    seq = ++sinfo->seq;
                }
                rc = rx::kv_pool_write_rows(desc, nb, (const int32_t*)(hm + L->off_prefix_slots),
                                            (const int64_t*)(hm + L->off_prefix_indptr),
                                            (const int32_t*)(hm + L->off_new_slots), (const int64_t*)(hm + L->off_qo_indptr),
                                            io->d_k_new, io->d_v_new, io->d_k_pool, io->d_v_pool, r2t_c, L->stride, t0, t1,
                                            io->d_status, stream, h_dev, io->d_stage, L->bytes,
                                            by_flag ? sinfo->ctr_dev : nullptr, by_flag ? sinfo->flag_dev : nullptr, seq);
                if (rc == RX_OK && by_flag) {
                    std::lock_guard<std::mutex> lk(g_ev_mu);
                    sinfo->mode = 2;
                } else if (rc == RX_OK) {
                    if (cudaEventRecord(ev, stream) != cudaSuccess) {
                        set_error("rx_step_launch: cannot record the staging event");
                        return RX_ECUDA;
                    }
                    std::lock_guard<std::mutex> lk(g_ev_mu);
                    sinfo->mode = 1;
                }
            } else {
                rc = rx::kv_pool_write_rows(desc, nb, prefix_slots, prefix_indptr + b0, new_slots, qo_indptr + b0,
                                            io->d_k_new, io->d_v_new, io->d_k_pool, io->d_v_pool, r2t_c, L->stride, t0,
                                            t1, io->d_status, stream);
            }
            if (rc != RX_OK) return rc;
            if (io->decode)   // decode rows are the requests themselves (one new token each)
                rc = decode_attention(desc, nb, (const char*)io->d_q + t0 * rb.q, r2t_c, L->stride, kv_lens + b0, gp,
                                      io->d_k_pool, io->d_v_pool, (char*)io->d_out + t0 * rb.q,
                                      io->d_lse ? io->d_lse + t0 * desc->hq : nullptr, L->max_kv_len, io->d_workspace,
                                      io->ws_bytes, io->d_status, stream);
            else
                rc = prefix_extend_attention(desc, nb, io->d_q, qo_indptr + b0, prefix_lens + b0, r2t_c, L->stride,
                                             io->d_k_pool, io->d_v_pool, io->d_out, io->d_lse, L->max_qo_len, gp,
                                             io->d_workspace, io->ws_bytes, io->d_status, stream);
            if (rc != RX_OK) return rc;
            if (!host) continue;
            // the output of these rows back to the host: behind the compute on the copy-out
            // stream when the step is ranged, else on `stream` itself
            cudaStream_t s_out = ranged ? pp->out : stream;
            if (ranged) {
                e = cudaEventRecord(pp->ev[3 + 2 * c], stream);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, pp->ev[3 + 2 * c], 0);
            }
            if (e == cudaSuccess)
                e = cudaMemcpyAsync((char*)io->h_out + t0 * rb.q, (const char*)io->d_out + t0 * rb.q,
                                    (size_t)((t1 - t0) * rb.q), cudaMemcpyDeviceToHost, s_out);
            if (e == cudaSuccess && io->h_lse && io->d_lse)
                e = cudaMemcpyAsync(io->h_lse + t0 * desc->hq, io->d_lse + t0 * desc->hq, (size_t)((t1 - t0) * desc->hq * 4),
                                    cudaMemcpyDeviceToHost, s_out);
        }
        if (e == cudaSuccess && host) {   // the step's kernels are done with its input rows
            cudaEvent_t r = nullptr;
            e = release_slot(pp->rel, 4, &pp->rel_next, io->d_q, &r);
            if (e == cudaSuccess) e = cudaEventRecord(r, stream);
        }
        if (e == cudaSuccess && sp) {     // ... and with its device staging buffer
            cudaEvent_t r = nullptr;
            e = release_slot(sp->srel, 4, &sp->srel_next, io->d_stage, &r);
            if (e == cudaSuccess) e = cudaEventRecord(r, stream);
        }
        if (e == cudaSuccess && host && ranged) {   // `stream` completes only after the last output copy
            e = cudaEventRecord(pp->ev[1], pp->out);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, pp->ev[1], 0);
        }
        if (e != cudaSuccess) {
            set_error("rx_step_launch: %s", cudaGetErrorString(e));
            return RX_ECUDA;
        }
    }
    return rx_step_finish(t, B, tokens, tok_indptr, last_nodes, h_stage, L, evict_tokens, out_evicted);
}

extern "C" int rx_step_run(const rx_step_args* a) {
    RX_TRACE("rx_step_run");
    RX_REQUIRE(a, "rx_step_run: bad arguments");
    rx_radix* t = a->tree;
    const rx_attn_desc* desc = a->desc;
    const int32_t batch = a->batch;
    const int32_t* tokens = a->tokens;
    const int64_t* tok_indptr = a->tok_indptr;
    const int32_t* n_new = a->n_new;
    void* h_stage = a->h_stage;
    const rx_step_io* io = a->io;
    rx_node* out_last = a->out_last;
    rx_step_layout* out = a->out;
    void* stream = a->stream;
    RX_REQUIRE(t && desc && io && h_stage && out && tok_indptr && batch >= 0, "rx_step_run: bad arguments");
    int rc = RX_OK;
    if (io->h_q && batch > 0) {           // the first range's rows start crossing the link now
        rc = rx_step_prefetch(desc, batch, n_new, io, stream);
        if (rc != RX_OK) return rc;
    }
    rc = rx_stage_wait(h_stage);
    if (rc != RX_OK) return rc;
    rc = rx_step_plan(t, batch, tokens, tok_indptr, n_new, a->group_mode, a->heads_per_kv, a->min_shared, h_stage,
                      a->stage_cap, out_last, out);
    if (rc != RX_OK) return rc;
    if (out->batch > 0 && out->total_new > 0) {
        const size_t ws = rx_step_workspace_bytes(desc, out, io->decode);
        if (!io->d_stage || io->d_stage_bytes < (size_t)out->bytes || !io->d_r2t ||
            io->r2t_elems < (int64_t)out->batch * out->stride || (ws > 0 && (!io->d_workspace || io->ws_bytes < ws))) {
            set_error("rx_step_run: device buffers too small for this plan (staging %zu of %lld, slot table %lld of "
                      "%lld, workspace %zu of %zu): planned, not launched",
                      io->d_stage_bytes, (long long)out->bytes, (long long)io->r2t_elems,
                      (long long)out->batch * out->stride, io->ws_bytes, ws);
            return RX_ENOMEM;
        }
    }
    return rx_step_launch(t, desc, tokens, tok_indptr, out_last, h_stage, out, io, a->evict_tokens, a->out_evicted,
                          stream);
}

extern "C" int rx_step_ranges(const rx_attn_desc* desc, int32_t batch, const int32_t* n_new, int32_t chunks,
                              int32_t* out_cuts, int32_t cap, int32_t* out_n) {
    RX_REQUIRE(desc && batch >= 0 && (batch == 0 || n_new) && out_cuts && out_n && cap > 0,
               "rx_step_ranges: bad arguments");
    RX_REQUIRE(desc->hq > 0 && desc->hkv > 0 && desc->head_dim > 0, "rx_step_ranges: bad descriptor");
    std::vector<int64_t> qo((size_t)batch + 1, 0);
    for (int32_t b = 0; b < batch; ++b) {
        RX_REQUIRE(n_new[b] >= 0, "rx_step_ranges: request %d has %d new tokens", b, n_new[b]);
        qo[(size_t)b + 1] = qo[(size_t)b] + n_new[b];
    }
    const std::vector<int32_t> cut = range_cuts(desc, qo.data(), batch, chunks);
    RX_REQUIRE((int64_t)cut.size() <= cap, "rx_step_ranges: %zu cut points, capacity %d", cut.size(), cap);
    std::copy(cut.begin(), cut.end(), out_cuts);
    *out_n = (int32_t)cut.size() - 1;
    return RX_OK;
}

extern "C" int rx_step_prefetch(const rx_attn_desc* desc, int32_t batch, const int32_t* n_new, const rx_step_io* io,
                                void* stream_) {
    RX_TRACE("rx_step_prefetch");
    RX_REQUIRE(desc && io && batch >= 0 && (batch == 0 || n_new), "rx_step_prefetch: bad arguments");
    RX_REQUIRE(io->h_q && io->h_k_new && io->h_v_new && io->d_q && io->d_k_new && io->d_v_new,
               "rx_step_prefetch: needs the host and device rows");
    std::vector<int64_t> qo((size_t)batch + 1, 0);
    for (int32_t b = 0; b < batch; ++b) {
        RX_REQUIRE(n_new[b] >= 0, "rx_step_prefetch: request %d has %d new tokens", b, n_new[b]);
        qo[(size_t)b + 1] = qo[(size_t)b] + n_new[b];
    }
    const std::vector<int32_t> cut = range_cuts(desc, qo.data(), batch, io->chunks);
    Pipe* pp = nullptr;
    int rc = pipe_for(2 + 2 * ((int)cut.size() - 1), &pp);
    if (rc != RX_OK) return rc;
    std::lock_guard<std::mutex> lk(pp->use);
    // the first range only: further copies would queue the step's index arrays behind them
    rc = copy_in(pp, desc, io, qo.data(), cut, 0, 1, true, (cudaStream_t)stream_);
    if (rc != RX_OK) return rc;
    pp->pending = true;
    pp->p_hq = io->h_q;
    pp->p_dq = io->d_q;
    pp->p_T = qo[(size_t)batch];
    pp->p_cut = cut;
    return RX_OK;
}
