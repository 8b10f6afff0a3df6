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
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "radix_attn.h"
#include "rx_common.h"

namespace {

std::mutex g_ev_mu;
std::unordered_map<const void*, cudaEvent_t> g_stage_events;   // staging buffer -> event of its last copy

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

extern "C" int rx_stage_wait(const void* h_stage) {
    cudaEvent_t ev = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ev_mu);
        auto it = g_stage_events.find(h_stage);
        if (it != g_stage_events.end()) ev = it->second;
    }
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
        cudaEvent_t ev = nullptr;
        {
            std::lock_guard<std::mutex> lk(g_ev_mu);
            auto it = g_stage_events.find(h_stage);
            if (it == g_stage_events.end()) {
                if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
                    set_error("rx_step_launch: cannot create an event");
                    return RX_ECUDA;
                }
                g_stage_events[h_stage] = ev;
            } else {
                ev = it->second;
            }
        }
        cudaError_t e = cudaMemcpyAsync(io->d_stage, h_stage, (size_t)L->bytes, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaEventRecord(ev, stream);
        if (e != cudaSuccess) {
            set_error("rx_step_launch: staging copy failed: %s", cudaGetErrorString(e));
            return RX_ECUDA;
        }
        unsigned char* ds = (unsigned char*)io->d_stage;
        const int32_t* prefix_slots = (const int32_t*)(ds + L->off_prefix_slots);
        const int64_t* prefix_indptr = (const int64_t*)(ds + L->off_prefix_indptr);
        const int32_t* new_slots = (const int32_t*)(ds + L->off_new_slots);
        const int64_t* qo_indptr = (const int64_t*)(ds + L->off_qo_indptr);
        const int32_t* prefix_lens = (const int32_t*)(ds + L->off_prefix_lens);
        const int32_t* kv_lens = (const int32_t*)(ds + L->off_kv_lens);
        int rc = kv_pool_write(desc, B, prefix_slots, prefix_indptr, new_slots, qo_indptr, io->d_k_new, io->d_v_new,
                               io->d_k_pool, io->d_v_pool, io->d_r2t, L->stride, L->total_new, io->d_status, stream);
        if (rc != RX_OK) return rc;
        rx_shared_groups g{};
        const rx_shared_groups* gp = nullptr;
        if (L->num_groups > 0) {
            g = groups_of(L, ds);
            gp = &g;
        }
        if (io->decode)
            rc = decode_attention(desc, B, io->d_q, io->d_r2t, L->stride, kv_lens, gp, io->d_k_pool, io->d_v_pool,
                                  io->d_out, io->d_lse, L->max_kv_len, io->d_workspace, io->ws_bytes, io->d_status, stream);
        else
            rc = prefix_extend_attention(desc, B, io->d_q, qo_indptr, prefix_lens, io->d_r2t, L->stride, io->d_k_pool,
                                         io->d_v_pool, io->d_out, io->d_lse, L->max_qo_len, gp, io->d_workspace,
                                         io->ws_bytes, io->d_status, stream);
        if (rc != RX_OK) return rc;
    }
    return rx_step_finish(t, B, tokens, tok_indptr, last_nodes, h_stage, L, evict_tokens, out_evicted);
}
