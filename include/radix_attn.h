/*
 * radix_attn.h -- C ABI of libradixattn.so: prefix-cached KV attention with a radix tree.
 *
 * The method: RadixAttention-style reuse of the KV cache across requests.
 *  - "SGLang: Efficient Execution of Structured Language Model Programs" (unite.ai), the
 *    RadixAttention bullet of the introduction: an LRU cache of KV kept in a radix tree,
 *    with matching, insertion and eviction; and the nine-step walk-through of the tree
 *    under an LRU policy (insert a turn as a node, reuse a cached prefix, split a node on
 *    partial sharing, evict least recently used nodes under memory pressure).
 *  - "Prompt Caching" (Ultralytics glossary), "How prompt caching works": with causal
 *    attention a token's keys/values depend only on earlier tokens, so a cached prefix's
 *    K/V can replace recomputation; only the new tokens run through the model; decode
 *    attends each new token to all cached keys/values.
 *
 * Conventions (every entry point):
 *  - Returns an int status (RX_OK or a negative RX_E* code); never throws or aborts.
 *    rx_last_error() gives a thread-local message for the last failure.
 *  - "d_" arguments are DEVICE pointers (caller-owned, e.g. torch tensors' data_ptr()),
 *    "h_"/plain pointer arguments are HOST pointers (caller-owned).  The library never
 *    allocates device memory; scratch space is passed in (decode workspace).
 *  - Device calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *    Launch errors return RX_ECUDA.  Data-dependent failures detected on the device (a
 *    slot out of range, a length beyond the table stride or a host hint) are written to
 *    *d_status (int32, first failure wins, 0 = ok) and the offending element is skipped;
 *    read it after synchronising.  Kernels never trap and never spin without a bound.
 *  - Token ids and slots are int32; lengths and offsets ("indptr") are int64 unless noted.
 *  - KV pools are [num_slots, hkv, head_dim], slot-major, row-contiguous, of the dtype in
 *    rx_attn_desc.  A request's slot table row req_to_token[b, 0:len] lists the pool slot
 *    of each of its tokens in logical order; unused entries are -1.
 *  - A radix tree is not thread-safe: use one tree per host thread or lock externally.
 */
#ifndef RADIX_ATTN_H
#define RADIX_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum rx_status {
    RX_OK = 0,
    RX_EINVAL = -1,    /* bad argument (null pointer, bad size, unknown handle, bad slot) */
    RX_ENOMEM = -2,    /* not enough free KV slots (nothing was allocated) */
    RX_ECUDA = -3,     /* a CUDA launch or runtime call failed */
    RX_ELOCKED = -4,   /* unlock of a node that is not locked */
    RX_ETIMEOUT = -5,  /* reserved: a bounded device wait gave up */
    RX_EDEVICE = -6    /* unsupported device or configuration (e.g. not sm_103a for a tcgen05 kernel) */
};

/* Codes written to *d_status by kernels. */
enum rx_device_status {
    RX_DEV_OK = 0,
    RX_DEV_BAD_SLOT = 1,     /* a slot outside [0, num_slots) was met; that row was skipped */
    RX_DEV_BAD_LENGTH = 2,   /* a length exceeds the table stride or the host hint; request skipped */
    RX_DEV_TIMEOUT = 3       /* a bounded wait inside a kernel gave up; outputs are invalid */
};

typedef enum { RX_F32 = 0, RX_BF16 = 1 } rx_dtype;

/* Shape of one attention layer.  hq % hkv == 0; query head h reads kv head h / (hq/hkv).
 * head_dim is 64 or 128.  scale multiplies q.k (1/sqrt(head_dim) in every workload). */
typedef struct {
    int32_t dtype;      /* rx_dtype of q, k, v, pools and outputs */
    int32_t hq;
    int32_t hkv;
    int32_t head_dim;
    int64_t num_slots;  /* rows of each KV pool */
    float scale;
} rx_attn_desc;

/* ========================================================================= radix tree
 * Host C++ radix tree mapping token sequences to KV-pool slots at token granularity,
 * plus the pool's slot allocator.  Readings the pages leave open:
 *  - a node boundary is cut at every divergence point and at the end of every match and
 *    insert; nodes never merge again;
 *  - a logical LRU clock advances by one per match_prefix/insert call and stamps every
 *    node on the touched path;
 *  - evict frees whole unlocked leaf nodes, least recent stamp first (ties by node id);
 *  - the free list is FIFO: alloc pops from the head, frees append to the tail; it starts
 *    as the slot ids ordered by the SplitMix64 output (state seed + (id+1)*0x9E3779B97F4A7C15,
 *    Steele/Lea/Flood 2014), ties by id. */
typedef struct rx_radix rx_radix;   /* opaque, host-owned */
typedef int64_t rx_node;            /* node handle; 0 = root */

typedef struct {
    int64_t match_calls;
    int64_t match_query_tokens;     /* tokens passed to match_prefix */
    int64_t match_hit_tokens;       /* tokens matched (the cache hits) */
    int64_t insert_calls;
    int64_t inserted_tokens;        /* tokens newly owned by the tree */
    int64_t evicted_tokens;
    int64_t node_count;             /* nodes excluding the root */
    int64_t cached_tokens;          /* tokens held by the tree */
    int64_t free_slots;
    int64_t num_slots;
} rx_stats;

/* Create a tree over a pool of num_slots slots (1 <= num_slots <= 2^31-1).
 * *out receives the tree; free it with radix_destroy. */
int radix_create(int64_t num_slots, uint64_t slot_perm_seed, rx_radix** out);
void radix_destroy(rx_radix* t);

/* Longest cached prefix of tokens[0:n].  Writes its slots to out_slots (capacity n),
 * its length to *out_len and the handle of the node ending there to *out_last (0 if none).
 * Splits the node in which the match ends and stamps the matched path. */
int match_prefix(rx_radix* t, const int32_t* tokens, int64_t n, int32_t* out_slots,
                 int64_t* out_len, rx_node* out_last);

/* Length of the longest cached prefix of tokens[0:n], read-only: no LRU stamp, no split, no
 * statistics.  A scheduler uses it to order waiting requests by how much of each is cached
 * (cache-aware scheduling, "SGLang: Efficient Execution of Structured Language Model
 * Programs", results on cache hit rates).  *out_len = the length match_prefix would return now. */
int match_prefix_len(const rx_radix* t, const int32_t* tokens, int64_t n, int64_t* out_len);

/* Reuse granularity (default 1 = token granular, as RadixAttention keeps it): with a page
 * size p > 1, every match (match_prefix, match_prefix_batch, match_prefix_len, rx_step_plan)
 * counts whole pages only -- the cached prefix cut down to a multiple of p, ending (split,
 * stamped) at that page boundary -- as a cache of fixed-size pages can reuse only full pages
 * (the aiezz OpenJev-on-SGLang tutorial, advanced serving tips, the tip on treating cache
 * reuse as an opportunity: cache page boundaries are one of the things that cut hits).
 * Storage stays token granular: the tail of a partly matched page is recomputed and its new
 * slots are returned as duplicates when inserted.
 * RX_EINVAL outside [1, 2^20]. */
int radix_set_page_size(rx_radix* t, int64_t page_size);

/* match_prefix_len for `batch` requests: request b is tokens[tok_indptr[b] : tok_indptr[b+1]];
 * out_len has capacity batch. */
int match_prefix_len_batch(const rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                           int64_t* out_len);

/* Pin / unpin the path from the root to a node so that evict never frees it
 * (reference counted along the whole path).  RX_ELOCKED if unlocking an unlocked node. */
int radix_lock(rx_radix* t, rx_node node);
int radix_unlock(rx_radix* t, rx_node node);

/* Lock / unlock n nodes, as n radix_lock / radix_unlock calls (an in-flight batch pins the
 * prefixes it matched so that eviction during the step cannot free them).  The lock batch
 * checks every handle first and changes nothing on an unknown one; the unlock batch stops
 * at the first node that is not locked (RX_ELOCKED). */
int radix_lock_batch(rx_radix* t, const rx_node* nodes, int32_t n);
int radix_unlock_batch(rx_radix* t, const rx_node* nodes, int32_t n);

/* Pop n free slots (FIFO) into out_slots; RX_ENOMEM and nothing taken if fewer are free.
 * Never evicts on its own: the caller calls evict and retries. */
int alloc_slots(rx_radix* t, int64_t n, int32_t* out_slots);

/* Return caller-held slots to the tail of the free list, in order.  RX_EINVAL (and no
 * change) if a slot is out of range, already free or repeated. */
int free_slots(rx_radix* t, const int32_t* slots, int64_t n);

/* Insert tokens[0:n] with their slots.  Positions already cached keep the tree's slots:
 * *out_dup_len receives how many leading positions were already present, and the caller
 * still owns (and should free) slots[0:dup_len]; the tree takes slots[dup_len:n].
 * *out_last receives the handle of the node ending at n. */
int insert(rx_radix* t, const int32_t* tokens, const int32_t* slots, int64_t n,
           int64_t* out_dup_len, rx_node* out_last);

/* Free unlocked least-recently-used leaf nodes until at least num_tokens tokens are freed
 * or nothing is evictable.  Freed slots go to the tail of the free list, node by node in
 * position order; the first `cap` of them are also written to out_freed (may be NULL).
 * *out_n receives the number of slots freed (may exceed num_tokens and cap). */
int evict(rx_radix* t, int64_t num_tokens, int32_t* out_freed, int64_t cap, int64_t* out_n);

/* Batched forms of match_prefix / insert for a batch of requests, processed in order
 * b = 0..batch-1 with exactly the semantics (and LRU clock ticks) of one call each.
 * Request b's tokens are tokens[tok_indptr[b] : tok_indptr[b+1]] (tok_indptr: [batch+1]).
 * match_prefix_batch packs the matched slots: request b's are
 * out_slots[out_indptr[b] : out_indptr[b+1]] (out_slots capacity tok_indptr[batch],
 * out_indptr [batch+1]), ready to pass to kv_pool_write as the prefix slots and indptr.
 * insert_batch takes one slot per token (same indptr) and returns dup lengths per request. */
int match_prefix_batch(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                       int32_t* out_slots, int64_t* out_indptr, rx_node* out_last);
int insert_batch(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                 const int32_t* slots, int64_t* out_dup_len, rx_node* out_last);

/* Insert continued from where each request's match ended: request b's full prompt is
 * tokens[tok_indptr[b] : tok_indptr[b+1]], its cached path ends at node nodes[b] (the
 * out_last of its match, still cached -- e.g. locked) at depth d_b, and new_slots[
 * new_indptr[b] : new_indptr[b+1]] holds one slot for each of its n_b - d_b later tokens.
 * Same result, stamps and dup lengths (counted from position 0) as insert of the full
 * prompt with the matched slots followed by the new ones, without re-walking the cached
 * prefix.  The caller owns new slots [0, dup_len - d_b) of a request (cached meanwhile). */
int insert_batch_at(rx_radix* t, int32_t batch, const rx_node* nodes, const int32_t* tokens,
                    const int64_t* tok_indptr, const int32_t* new_slots, const int64_t* new_indptr,
                    int64_t* out_dup_len, rx_node* out_last);

/* ------------------------------------------------------------------ step runtime
 * One serving step over a batch of prompts, with all host work native: rx_step_plan does
 * a1/a2 (match, allocate, pin) and lays every index array the kernels need into a
 * caller-provided staging buffer (pinned host memory, copied to the device with one
 * transfer); rx_step_finish does a7/a8 (insert, evict) and unpins.  Offsets are bytes from
 * the start of the staging buffer, each 256-byte aligned; the same offsets apply to the
 * device copy.  Arrays: prefix_slots int32 [sum P_b], prefix_indptr int64 [batch+1],
 * new_slots int32 [T], qo_indptr int64 [batch+1], prefix_lens int32 [batch], kv_lens int32
 * [batch] (P_b + n_b), and with groups grp_indptr / grp_members / grp_len int32. */
typedef struct {
    int32_t batch;
    int32_t max_qo_len, max_kv_len, stride;  /* stride = max_kv_len rounded up to 8 */
    int64_t total_new;                       /* T */
    int64_t total_prefix;                    /* sum P_b */
    int64_t bytes;                           /* bytes of the staging buffer in use */
    int64_t off_prefix_slots, off_prefix_indptr, off_new_slots, off_qo_indptr, off_prefix_lens, off_kv_lens;
    int32_t num_groups, max_group_size, max_group_len, max_group_rows;
    int64_t off_grp_indptr, off_grp_members, off_grp_len;
} rx_step_layout;

enum { RX_GROUPS_NONE = 0, RX_GROUPS_ALWAYS = 1, RX_GROUPS_AUTO = 2 };

/* Upper bound of the staging bytes rx_step_plan needs for these prompts. */
size_t rx_step_stage_bytes(int32_t batch, int64_t total_tokens);

/* Plan one step: request b's prompt is tokens[tok_indptr[b] : tok_indptr[b+1]], of which the
 * last n_new[b] tokens must be uncached (RX_EINVAL otherwise, nothing allocated); allocates
 * their slots (RX_ENOMEM if short: evict and retry), locks each request's matched node
 * (out_last[b], capacity batch) until rx_step_finish.  group_mode: RX_GROUPS_NONE, _ALWAYS
 * (radix_shared_groups with min_shared) or _AUTO (only when every request is in a group, its
 * remaining keys are <= 256 and a request's new rows times heads_per_kv stay below 128 --
 * the shape where stacking rows pays -- and not when every request has at most 8 rows
 * (new tokens x heads_per_kv) over at most 1024 keys, which the small-extend kernel serves). */
int rx_step_plan(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                 const int32_t* n_new, int32_t group_mode, int32_t heads_per_kv, int64_t min_shared,
                 void* h_stage, size_t stage_cap, rx_node* out_last, rx_step_layout* out);

/* Finish the step planned into h_stage: insert every prompt from its matched node, return
 * new slots that turned out cached to the free list, evict >= evict_tokens LRU tokens (0:
 * none; *out_evicted receives the count, may be NULL) and unlock the matched nodes. */
int rx_step_finish(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                   const rx_node* last_nodes, const void* h_stage, const rx_step_layout* layout,
                   int64_t evict_tokens, int64_t* out_evicted);

int radix_stats(const rx_radix* t, rx_stats* out);

/* Check the tree's invariants (edges, parents, slot ownership, stamps, locks);
 * RX_OK or RX_EINVAL with the first violation in rx_last_error(). */
int radix_check(const rx_radix* t);

/* Shared-prefix groups for a decode batch, derived from the tree.  last_nodes[b] is the
 * node where request b's cached path ends (out_last of its match_prefix/insert).  Requests
 * whose paths leave the root through the same child node form one group; the group's
 * shared length is the token depth of the deepest node common to all of its members'
 * paths.  Groups with fewer than two members or a shared length below min_shared are not
 * formed.  out_group_of[b] = group id or -1 (capacity batch); out_group_len[g] = shared
 * tokens of group g (capacity batch); *out_num_groups = number of groups.  Group ids are
 * assigned in order of each group's first member. */
int radix_shared_groups(const rx_radix* t, const rx_node* last_nodes, int32_t batch,
                        int64_t min_shared, int32_t* out_group_of, int64_t* out_group_len,
                        int32_t* out_num_groups);

/* ========================================================================= kernels */

/* Build the slot table and scatter the new tokens' K/V into the pools.
 * For request b (0 <= b < batch):
 *   P_b = prefix_indptr[b+1]-prefix_indptr[b] matched slots d_prefix_slots[prefix_indptr[b]..],
 *   n_b = qo_indptr[b+1]-qo_indptr[b] new slots d_new_slots[qo_indptr[b]..];
 *   req_to_token[b, 0:P_b] = matched slots, [P_b:P_b+n_b] = new slots, rest = -1.
 *   For every new token t, k_pool[new_slots[t]] = k_new[t], v_pool[new_slots[t]] = v_new[t]
 *   (rows of hkv*head_dim elements).
 * d_k_new/d_v_new: [T, hkv, head_dim] with T = total_new = qo_indptr[batch] (host copy;
 * sizes the grid, and a request reaching past it is a length error).  d_req_to_token:
 * [batch, r2t_stride] int32.  P_b + n_b > r2t_stride -> RX_DEV_BAD_LENGTH for that row;
 * a slot outside [0, num_slots) -> RX_DEV_BAD_SLOT and that row is not written.
 * "Prompt Caching", "How prompt caching works": only the new tokens' K/V are computed and
 * stored; the prefix entries point at the cached copies. */
int kv_pool_write(const rx_attn_desc* desc, int32_t batch,
                  const int32_t* d_prefix_slots, const int64_t* d_prefix_indptr,
                  const int32_t* d_new_slots, const int64_t* d_qo_indptr,
                  const void* d_k_new, const void* d_v_new,
                  void* d_k_pool, void* d_v_pool,
                  int32_t* d_req_to_token, int64_t r2t_stride, int64_t total_new,
                  int32_t* d_status, void* stream);

/* Optional description of requests that share a leading run of KV (a cached prefix), for
 * decode_attention and prefix_extend_attention.  Members of group g have identical
 * req_to_token[b, 0:len_g] (e.g. radix_shared_groups on their matched nodes); the shared
 * part is read once per group, for all members' query rows stacked, instead of once per
 * member, and merged exactly with each member's private part. */
typedef struct {
    int32_t num_groups;
    int32_t max_group_size;          /* host hint: largest group (members) */
    const int32_t* d_group_indptr;   /* [num_groups+1] offsets into d_group_members */
    const int32_t* d_group_members;  /* request ids; a request is in at most one group */
    const int32_t* d_group_len;      /* [num_groups] shared leading tokens, >= 1 */
    int32_t max_group_len;           /* host hint: largest d_group_len */
    int32_t max_group_rows;          /* extend only, host hint: largest sum of new tokens over a group's members */
} rx_shared_groups;

/* Extend (prefill over the new tokens) attention with a cached prefix.
 * For request b with P_b = d_prefix_lens[b] cached tokens and n_b = qo_indptr[b+1]-qo_indptr[b]
 * new tokens, new row i (absolute position p = P_b + i) of query head h computes
 *   o = softmax(scale * q K[0..p]^T) V[0..p]
 * where K/V row j is the pool row req_to_token[b, j] of kv head h/(hq/hkv): the cached
 * prefix is gathered from its slots and the new tokens attend causally to themselves
 * (self included).  "Prompt Caching", "How prompt caching works" (causal attention; the
 * cached prefix replaces recomputation).
 * d_q, d_out: [T, hq, head_dim]; d_lse: optional [T, hq] float32 natural-log log-sum-exp
 * of the scaled scores.  max_qo_len (host) must be >= every n_b (sizes the grid); rows of
 * a request with n_b > max_qo_len or P_b + n_b > r2t_stride are skipped with
 * RX_DEV_BAD_LENGTH.  bf16 runs on tcgen05 tensor cores (sm_103a); f32 on CUDA cores.
 * groups (optional, bf16): requests sharing a cached prefix.  Their new rows are stacked
 * into dense tiles against one read of the shared run (tcgen05), each request's remaining
 * keys (its private cached tokens and its new tokens, causally) are done per row on CUDA
 * cores, and the two softmax parts are merged exactly.  Worth it when the new rows per
 * request are few and the private parts short (e.g. many short questions on one system
 * prompt).  d_workspace: >= extend_workspace_bytes(...) bytes, 256-byte aligned, needed only
 * with groups (else NULL / 0).  bf16 calls take at most 65535 requests and, on the tcgen05
 * kernel, max_qo_len * hq/hkv below 65536 * 256 (RX_EINVAL beyond: split the batch). */
int prefix_extend_attention(const rx_attn_desc* desc, int32_t batch,
                            const void* d_q, const int64_t* d_qo_indptr, const int32_t* d_prefix_lens,
                            const int32_t* d_req_to_token, int64_t r2t_stride,
                            const void* d_k_pool, const void* d_v_pool,
                            void* d_out, float* d_lse, int32_t max_qo_len,
                            const rx_shared_groups* groups, void* d_workspace, size_t ws_bytes,
                            int32_t* d_status, void* stream);

/* Bytes of device workspace prefix_extend_attention needs with these groups (0 without). */
size_t extend_workspace_bytes(const rx_attn_desc* desc, int32_t batch, int32_t max_qo_len,
                              const rx_shared_groups* groups);

/* Bytes of device workspace decode_attention needs for this batch (>= 0), or 0 on error. */
size_t decode_workspace_bytes(const rx_attn_desc* desc, int32_t batch, int32_t max_kv_len,
                              const rx_shared_groups* groups);

/* Decode attention: one query token per request attends all of its L_b = d_kv_lens[b]
 * cached tokens (the new token's own K/V must already be in the pool, e.g. by
 * kv_pool_write): o = softmax(scale * q K[0..L_b-1]^T) V[0..L_b-1] per query head.
 * "Prompt Caching", "How prompt caching works": in decode each new token attends to all
 * cached keys and values.  The keys are split into chunks processed by different CTAs
 * (split-KV); per-chunk partial results (normalised output and log-sum-exp) are merged
 * by a second kernel.  With `groups`, a group's shared leading tokens are processed once
 * for all its members (their query rows stacked into one tile) and merged with each
 * member's private remainder.
 * d_q, d_out: [batch, hq, head_dim]; d_lse optional [batch, hq] float32.
 * max_kv_len (host) must be >= every L_b.  d_workspace: >= decode_workspace_bytes(...)
 * bytes of device memory, contents need not be initialised.  The requests are a launch
 * dimension of the bf16 kernels: a call takes at most 65535 of them (more fail to launch and
 * return RX_ECUDA with the launch error in rx_last_error); larger batches are split by the
 * caller. */
int decode_attention(const rx_attn_desc* desc, int32_t batch,
                     const void* d_q, const int32_t* d_req_to_token, int64_t r2t_stride,
                     const int32_t* d_kv_lens, const rx_shared_groups* groups,
                     const void* d_k_pool, const void* d_v_pool,
                     void* d_out, float* d_lse, int32_t max_kv_len,
                     void* d_workspace, size_t ws_bytes,
                     int32_t* d_status, void* stream);

/* decode_attention without a caller-provided workspace.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory per call -- a
 * plug-in inside a host application whose allocator already owns the GPU's memory, a
 * serving loop that must not stall on cudaMalloc/cudaFree (they can synchronise the
 * device), or a plain C caller with no allocator to provide the workspace.  The split-KV
 * scratch lives in one static device array of RX_DECODE_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library holds until the process exits; nothing is allocated per call.
 *  - Arguments and results are those of decode_attention (inputs and outputs are still the
 *    caller's buffers).
 *  - A batch whose decode_workspace_bytes(...) exceeds RX_DECODE_NOALLOC_SCRATCH_BYTES is
 *    rejected with RX_EINVAL and a message; split the batch or use decode_attention.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress, a host-side lookup), so the address stays right after a
 *    cudaDeviceReset or on another device.  The first call on a device may load the
 *    library's device code there; make that first call before any stream capture.
 *  - All calls share the one array (it keeps the last call's contents; every call writes
 *    the scratch before reading it): calls that overlap on the GPU -- on different streams,
 *    or from different host threads -- race and give wrong results.  Serialise them. */
#define RX_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)
int decode_attention_noalloc(const rx_attn_desc* desc, int32_t batch,
                             const void* d_q, const int32_t* d_req_to_token, int64_t r2t_stride,
                             const int32_t* d_kv_lens, const rx_shared_groups* groups,
                             const void* d_k_pool, const void* d_v_pool,
                             void* d_out, float* d_lse, int32_t max_kv_len,
                             int32_t* d_status, void* stream);

/* ------------------------------------------------------------------ one-call step launch
 * Everything of a planned step that follows rx_step_plan, in one call: the staging buffer
 * (h_stage) to its device copy (io->d_stage) -- for at most 1 MiB of device-row step, by
 * kv_pool_write's own launch reading the device mapping of the pinned buffer; in host-buffer
 * mode a kernel reading that mapping; else a copy-engine transfer --, kv_pool_write (a3), the
 * attention -- prefix_extend_attention (a4), or decode_attention (a5/a6) when io->decode --
 * with the plan's shared-prefix groups, and rx_step_finish (a7/a8: insert, free duplicates,
 * evict evict_tokens, unpin; host only, it does not wait for the GPU).  All device work is
 * enqueued on `stream`.  Device buffers are the caller's: the rows of the step's new tokens
 * (d_q, d_k_new, d_v_new: [T, hq|hkv, head_dim] in qo_indptr order), d_out (and optional
 * d_lse), the pools, d_stage (>= layout bytes), d_r2t (>= batch * stride int32) and
 * d_workspace (>= rx_step_workspace_bytes).  After the call the staging buffer is still
 * being read by the copy: call rx_stage_wait(h_stage) before planning into it again.
 * Host-buffer mode (h_q set): the step's new rows come from host memory -- h_q, h_k_new,
 * h_v_new in the layout of d_q, d_k_new, d_v_new (pinned, for the copies to run
 * asynchronously) -- and the output goes back to h_out (and h_lse, optional).  The requests
 * are cut into `chunks` ranges of about equal token counts (0: chosen from the bytes moved, and
 * with several ranges the last eighth of the last range's tokens becomes a range of its own, so
 * that the one output copy no later kernel hides is short) that run as a pipeline on two
 * internal copy streams: the rows of range c+1 are copied in while range c computes on
 * `stream` and the output of range c-1 is copied out (with shared-prefix groups the rows still
 * cross in ranges, and one computation over all of them starts once every range is in).  `stream` waits for the last copy, so the host buffers are complete (and
 * may be reused) once `stream` is.  The device buffers are still the caller's.  The input
 * copies wait for all work already on `stream`, or, with io->overlap set, only for the
 * kernels of the last host-buffer step whose d_q was this step's d_q (when the library still
 * tracks it: it keeps the last four; an untracked d_q waits for all work on `stream`).  With
 * overlap the caller must have no other reads of d_q, d_k_new or d_v_new pending on `stream`;
 * a caller that uses two sets of device input rows in turn then gets the copies of a step
 * running under the kernels of the previous one.
 * Returns RX_EINVAL (nothing launched, the plan still pinned) when a buffer is too small;
 * a launch failure returns RX_ECUDA; *out_evicted (may be NULL) receives the evicted count. */
typedef struct {
    const void* d_q;
    const void* d_k_new;
    const void* d_v_new;
    void* d_k_pool;
    void* d_v_pool;
    void* d_out;
    float* d_lse;                 /* optional */
    void* d_stage;
    size_t d_stage_bytes;
    int32_t* d_r2t;
    int64_t r2t_elems;
    void* d_workspace;
    size_t ws_bytes;
    int32_t* d_status;
    int32_t decode;               /* 1: one new token per request, decode_attention */
    const void* h_q;              /* host-buffer mode: NULL for device rows already filled */
    const void* h_k_new;
    const void* h_v_new;
    void* h_out;
    float* h_lse;                 /* optional */
    int32_t chunks;               /* host-buffer mode: request ranges of the pipeline (0: auto) */
    int32_t overlap;              /* 1: host-buffer mode, the input copies wait only for the last
                                     step that read the same d_q (see above); device rows, the
                                     index arrays are copied on an internal copy stream after
                                     the kernels of the last step that read the same d_stage
                                     (tracked as for d_q), and `stream` waits for the copy --
                                     with two d_stage buffers in turn, under the previous
                                     step's kernels */
} rx_step_io;

size_t rx_step_workspace_bytes(const rx_attn_desc* desc, const rx_step_layout* layout, int32_t decode);
int rx_step_launch(rx_radix* t, const rx_attn_desc* desc, const int32_t* tokens, const int64_t* tok_indptr,
                   const rx_node* last_nodes, void* h_stage, const rx_step_layout* layout, const rx_step_io* io,
                   int64_t evict_tokens, int64_t* out_evicted, void* stream);
/* Host-buffer mode: start the copies of a step's new rows (io->h_q, h_k_new, h_v_new into
 * io->d_q, d_k_new, d_v_new) before the step is planned, so that they overlap the plan: the
 * rows of the pipeline's first request range (rx_step_launch copies the others after the
 * step's index arrays, which would otherwise queue behind them).
 * Request b's rows are n_new[b] consecutive rows after those of requests 0..b-1 (the plan's
 * qo order), so the pipeline's request ranges (io->chunks, 0: automatic) follow from n_new
 * alone.  The copies run after the work already on `stream` (with io->overlap: after the
 * kernels of the last step that read io->d_q, as in rx_step_launch).  The next host-buffer
 * rx_step_launch on this device with the same h_q and d_q uses them instead of copying again
 * (RX_EINVAL if its plan has other row counts); no other host-buffer step may run on the
 * device in between. */
int rx_step_prefetch(const rx_attn_desc* desc, int32_t batch, const int32_t* n_new, const rx_step_io* io,
                     void* stream);

/* The request ranges a host-buffer step with these new-token counts is cut into (the same
 * cuts rx_step_prefetch and rx_step_launch make; a host computation, no device needed; no
 * counterpart on the pages: it exposes the pipeline's sizing for callers and tests).  Writes
 * the n+1 cut points (request indices, first 0, last batch) to out_cuts (capacity cap) and n
 * to *out_n.  n_new: host, [batch], each >= 0; chunks as rx_step_io.chunks.  RX_EINVAL on bad
 * arguments or too small a capacity (max(chunks, 4) + 2 entries always suffice). */
int rx_step_ranges(const rx_attn_desc* desc, int32_t batch, const int32_t* n_new, int32_t chunks, int32_t* out_cuts,
                   int32_t cap, int32_t* out_n);

/* Block until the last rx_step_launch that read h_stage is done with it (no-op if none): by
 * its CUDA event, or, for a small device-row step (index arrays read by kv_pool_write itself
 * through the buffer's device mapping), by a sequence number that launch writes to pinned host
 * memory when its last block is done -- read here without a CUDA call while the GPU is ahead;
 * after that, with short sleeps, returning RX_ECUDA on a context fault or after 60 s. */
int rx_stage_wait(const void* h_stage);

/* A whole step in one call, for a serving loop that crosses the library boundary once per
 * step (the pages' serving step: match the cached prefix, compute only the new tokens,
 * insert them -- "SGLang: Efficient Execution of Structured Language Model Programs",
 * RadixAttention and the nine-step walk-through).  The arguments sit in one struct, so that a
 * loop keeps one per staging buffer and changes only the step's inputs (batch, tokens,
 * tok_indptr, n_new) between calls.  In order: in host-buffer mode (io->h_q set)
 * rx_step_prefetch; rx_stage_wait(h_stage); rx_step_plan(tree, batch, tokens, tok_indptr,
 * n_new, group_mode, heads_per_kv, min_shared, h_stage, stage_cap, out_last, out); then, when
 * io's device buffers hold the plan -- d_stage_bytes >= out->bytes, r2t_elems >= batch *
 * out->stride, ws_bytes >= rx_step_workspace_bytes(desc, out, io->decode) -- rx_step_launch
 * with evict_tokens (*out_evicted, may be NULL, gets the evicted count) on `stream`.  When a
 * device buffer is too small it returns RX_ENOMEM with the plan made and pinned and nothing
 * launched: the caller grows the buffer (sizes from *out) and completes the step with
 * rx_step_launch on that plan.  Any other failure is returned as the failing call returns it.
 * The struct is only read; *out, out_last and *out_evicted are written. */
typedef struct {
    rx_radix* tree;
    const rx_attn_desc* desc;
    int32_t batch;
    int32_t group_mode;           /* RX_GROUPS_NONE / _ALWAYS / _AUTO */
    const int32_t* tokens;        /* host, the prompts concatenated */
    const int64_t* tok_indptr;    /* host, [batch + 1] */
    const int32_t* n_new;         /* host, [batch] */
    int32_t heads_per_kv;
    int32_t pad0;
    int64_t min_shared;
    void* h_stage;                /* pinned staging buffer and its size in bytes */
    size_t stage_cap;
    const rx_step_io* io;
    int64_t evict_tokens;
    rx_node* out_last;            /* host, [batch] */
    rx_step_layout* out;
    int64_t* out_evicted;         /* optional */
    void* stream;                 /* cudaStream_t */
} rx_step_args;

int rx_step_run(const rx_step_args* args);

/* Thread-local message describing the last failure in this thread ("" if none). */
const char* rx_last_error(void);

/* Library version string. */
const char* rx_version(void);

/* Tracing (the pages have no counterpart; a profiling aid): on != 0 puts an NVTX range named
 * after the entry point around every call that does work (the tree operations, the step
 * runtime's plan/launch/finish/prefetch/stage wait, kv_pool_write and the attention calls), so
 * that a profiler's timeline shows the library's host and GPU work per call.  Off by default;
 * RX_NVTX=1 in the environment when the library is loaded turns it on from the start.  While
 * off, a call pays one relaxed atomic load.  Process-wide; returns the previous setting. */
int rx_set_tracing(int on);

/* Self-test of the bounded waits inside the kernels: one CTA waits on an mbarrier that no
 * thread arrives at; after limit_ns (clamped to [1 us, 100 ms]) the wait gives up and sets
 * *d_status (device int32, caller-owned) to RX_DEV_TIMEOUT unless it already holds a code, and
 * the kernel ends.  The device stays usable.  Asynchronous on `stream`; RX_ECUDA if the launch
 * fails. */
int rx_wait_selftest(int32_t* d_status, uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* RADIX_ATTN_H */
