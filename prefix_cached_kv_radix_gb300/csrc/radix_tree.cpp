// Host radix tree over KV-pool slots, with LRU eviction and a FIFO slot allocator.
//
// "SGLang: Efficient Execution of Structured Language Model Programs" (unite.ai):
//  - RadixAttention bullet of the introduction: the runtime keeps an LRU cache of KV cache
//    in a radix tree and uses it for matching, insertion and eviction;
//  - the nine-step walk-through: edges carry token sequences; a new turn is inserted as a
//    node; a prompt whose prefix is in the tree reuses that KV; an edge is split in two
//    when a new sequence shares only part of it; under memory limits the least recently
//    used nodes are evicted.
// "Prompt Caching" (Ultralytics glossary): reuse needs an exactly matching prefix.
//
// Design: token-granular edges (each token owns one pool slot), children keyed by their
// first token.  Readings where the pages are open: a boundary is cut at every divergence
// point and at the end of every match and insert, and nodes never merge; a logical clock
// (+1 per match/insert call) stamps every node on the touched path; eviction frees whole
// unlocked leaves, least recent stamp first, ties by node id; locks are reference counts
// held along the whole root path.  The allocator is a FIFO ring of free slots whose
// initial order sorts slot ids by SplitMix64 (Steele, Lea & Flood, OOPSLA 2014).
#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <new>
#include <queue>
#include <string>
#include <thread>
#include <tuple>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include <unistd.h>

#include "rx_common.h"

namespace rx {

static thread_local std::string g_last_error;

static int trace_from_env() {
    const char* e = std::getenv("RX_NVTX");
    return (e && e[0] == '1') ? 1 : 0;
}
std::atomic<int> g_trace{trace_from_env()};

void set_error(const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
}

void clear_error() { g_last_error.clear(); }

struct Node;

// Map from an integer key to a node (a null node marks an empty cell): open addressing with
// linear probing over a power-of-two table kept at most 3/4 full, a multiplicative hash, and
// deletion by backward shift (no tombstones).  Clearing keeps the table, so a reused node's
// child map allocates nothing.  The tree's child links (by first token) and node handles
// (by id) live in these: a lookup is one multiply and, mostly, one cache line.
template <class K>
class NodeMap {
  public:
    Node* find(K k) const {
        if (n_ == 0) return nullptr;
        for (size_t i = home(k);; i = (i + 1) & mask_) {
            const Cell& c = cells_[i];
            if (!c.val) return nullptr;
            if (c.key == k) return c.val;
        }
    }
    void set(K k, Node* v) {   // insert, or replace the node of k
        if ((n_ + 1) * 4 > cells_.size() * 3) grow();
        size_t i = home(k);
        for (; cells_[i].val; i = (i + 1) & mask_)
            if (cells_[i].key == k) {
                cells_[i].val = v;
                return;
            }
        cells_[i] = Cell{k, v};
        ++n_;
    }
    bool erase(K k) {
        if (n_ == 0) return false;
        size_t i = home(k);
        for (; cells_[i].val; i = (i + 1) & mask_)
            if (cells_[i].key == k) break;
        if (!cells_[i].val) return false;
        // backward shift: an entry after the hole moves into it unless its home lies in the
        // cyclic range (hole, entry]
        for (size_t j = (i + 1) & mask_; cells_[j].val; j = (j + 1) & mask_) {
            const size_t h = home(cells_[j].key);
            const bool stays = i <= j ? (i < h && h <= j) : (i < h || h <= j);
            if (!stays) {
                cells_[i] = cells_[j];
                i = j;
            }
        }
        cells_[i].val = nullptr;
        --n_;
        return true;
    }
    size_t size() const { return n_; }
    bool empty() const { return n_ == 0; }
    void clear() {
        if (n_ == 0) return;
        for (Cell& c : cells_) c.val = nullptr;
        n_ = 0;
    }
    template <class F>
    void for_each(F&& f) const {
        for (const Cell& c : cells_)
            if (c.val) f(c.key, c.val);
    }

  private:
    struct Cell {
        K key;
        Node* val;
    };
    size_t home(K k) const { return (size_t)(((uint64_t)k * 0x9E3779B97F4A7C15ull) >> shift_); }
    void grow() {
        std::vector<Cell> old;
        old.swap(cells_);
        const size_t cap = old.empty() ? 4 : old.size() * 2;
        cells_.assign(cap, Cell{K(), nullptr});
        mask_ = cap - 1;
        shift_ = 64;
        for (size_t c = cap; c > 1; c >>= 1) --shift_;
        n_ = 0;
        for (const Cell& c : old)
            if (c.val) set(c.key, c.val);
    }
    std::vector<Cell> cells_;
    size_t mask_ = 0, n_ = 0;
    unsigned shift_ = 64;
};

struct Node {
    int64_t id = 0;
    Node* parent = nullptr;
    std::vector<int32_t> key;     // edge tokens
    std::vector<int32_t> slots;   // pool slot of each edge token
    NodeMap<int32_t> children;    // by first token
    uint64_t stamp = 0;
    int64_t ref = 0;
    int64_t depth = 0;            // tokens from the root to the END of this node
};

static uint64_t splitmix64_at(uint64_t seed, uint64_t counter) {
    uint64_t z = seed + counter * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// A small persistent pool for the data-parallel parts of a step's host work: reading every
// prompt against the tree and copying matched slots.  Those tasks only read the tree, one
// per request.  run(n, fn) calls fn(i) for every i in [0, n) on the workers and the calling
// thread and returns when all calls are done; one parallel region runs at a time (a
// concurrent caller runs its loop alone), and a process forked after the workers started
// (which has none of them) runs every loop alone.
class Pool {
  public:
    static Pool& get() {
        static Pool* p = new Pool();   // never destroyed: idle workers just wait
        return *p;
    }
    void run(int64_t n, const std::function<void(int64_t)>& fn) {
        std::unique_lock<std::mutex> region(call_, std::try_to_lock);
        if (!region.owns_lock() || workers_.empty() || n < 2 || getpid() != owner_) {
            for (int64_t i = 0; i < n; ++i) fn(i);
            return;
        }
        {
            std::lock_guard<std::mutex> g(m_);
            fn_ = &fn;
            n_ = n;
            next_.store(0);
            busy_ = (int)workers_.size();
            ++gen_;
        }
        cv_.notify_all();
        drain();
        std::unique_lock<std::mutex> g(m_);
        done_cv_.wait(g, [&] { return busy_ == 0; });
        fn_ = nullptr;
    }

  private:
    Pool() : owner_(getpid()) {
        const unsigned hc = std::thread::hardware_concurrency();
        const unsigned nw = hc > 1 ? std::min(7u, hc - 1) : 0u;
        for (unsigned i = 0; i < nw; ++i) {
            try {
                workers_.emplace_back([this] { loop(); });
            } catch (...) {
                break;                 // fewer workers (the caller always takes part)
            }
        }
        for (auto& w : workers_) w.detach();
    }
    void drain() {
        for (int64_t i = next_.fetch_add(1); i < n_; i = next_.fetch_add(1)) (*fn_)(i);
    }
    void loop() {
        uint64_t seen = 0;
        for (;;) {
            {
                std::unique_lock<std::mutex> g(m_);
                cv_.wait(g, [&] { return gen_ != seen; });
                seen = gen_;
            }
            drain();
            std::lock_guard<std::mutex> g(m_);
            if (--busy_ == 0) done_cv_.notify_one();
        }
    }
    const pid_t owner_;
    std::vector<std::thread> workers_;
    std::mutex call_, m_;
    std::condition_variable cv_, done_cv_;
    const std::function<void(int64_t)>* fn_ = nullptr;
    int64_t n_ = 0;
    std::atomic<int64_t> next_{0};
    int busy_ = 0;
    uint64_t gen_ = 0;
};

// Prompts shorter than this in total are read on the calling thread alone.
constexpr int64_t kParallelTokens = 1 << 15;

// Length of the common prefix of a[0:n] and b[0:n], starting the search at `from`.  Long
// equal runs (the common case: a prompt along a cached edge) go 64 tokens at a time through
// memcmp, the C library's vector compare (2-3x the rate of the loop below); then blocks of 16
// are OR-reduced, which the compiler vectorises, and the mismatch is found token by token.
static inline int64_t common_prefix(const int32_t* a, const int32_t* b, int64_t from, int64_t n) {
    int64_t k = from;
    while (k + 64 <= n && std::memcmp(a + k, b + k, 64 * sizeof(int32_t)) == 0) k += 64;
    while (k + 16 <= n) {
        uint32_t acc = 0;
        for (int i = 0; i < 16; ++i) acc |= (uint32_t)(a[k + i] ^ b[k + i]);
        if (acc) break;
        k += 16;
    }
    while (k < n && a[k] == b[k]) ++k;
    return k;
}

}  // namespace rx

struct rx_radix {
    int64_t num_slots = 0;
    // FIFO ring of free slots
    std::vector<int32_t> ring;
    int64_t head = 0, count = 0;
    std::vector<uint8_t> is_free;
    rx::Node root;
    uint64_t clock = 0;
    int64_t next_id = 1;
    int64_t page = 1;                  // reuse granularity: matches count whole pages only
    rx::NodeMap<int64_t> by_id;        // node handles
    rx_stats st{};

    // Evicted nodes, kept for reuse: a node's edge vectors and child map keep their capacity,
    // so the steady state of insert and evict (a step's leaves in, an older step's out)
    // allocates nothing.  At most kSpareNodes are kept.
    static constexpr size_t kSpareNodes = 4096;
    std::vector<rx::Node*> spare;
    // evict's scratch (the walk's stack and the heap of evictable leaves), kept between calls
    using EvictItem = std::tuple<uint64_t, int64_t, rx::Node*>;
    std::vector<rx::Node*> ev_stack;
    std::vector<EvictItem> ev_heap;
    void add_child(rx::Node* parent, int32_t tok, rx::Node* c) { parent->children.set(tok, c); }
    void drop_child(rx::Node* parent, int32_t tok) { parent->children.erase(tok); }
    void add_id(int64_t id, rx::Node* n) { by_id.set(id, n); }
    void drop_id(int64_t id) { by_id.erase(id); }

    ~rx_radix() {
        destroy_children(&root);
        for (rx::Node* n : spare) delete n;
    }

    void destroy_children(rx::Node* x) {
        std::vector<rx::Node*> stack;
        x->children.for_each([&](int32_t, rx::Node* c) { stack.push_back(c); });
        x->children.clear();
        while (!stack.empty()) {
            rx::Node* n = stack.back();
            stack.pop_back();
            n->children.for_each([&](int32_t, rx::Node* c) { stack.push_back(c); });
            delete n;
        }
    }

    // The free list is a ring of num_slots entries from `head`; positions wrap without a
    // division per slot.
    int64_t ring_pos(int64_t i) const {
        const int64_t p = head + i;
        return p < num_slots ? p : p - num_slots;
    }

    void push_free(int32_t s) {
        ring[(size_t)ring_pos(count)] = s;
        ++count;
        is_free[s] = 1;
    }

    rx::Node* new_node() {
        rx::Node* n;
        if (!spare.empty()) {
            n = spare.back();
            spare.pop_back();
            n->parent = nullptr;
            n->key.clear();
            n->slots.clear();
            n->children.clear();
            n->stamp = 0;
            n->ref = 0;
            n->depth = 0;
        } else {
            n = new rx::Node();
        }
        n->id = next_id++;
        add_id(n->id, n);
        ++st.node_count;
        return n;
    }

    // Split node c after its first k tokens.  The new upper node takes the first k tokens
    // and a new id; c keeps its id (a handle keeps naming the node that ends where it did).
    rx::Node* split(rx::Node* c, size_t k) {
        rx::Node* top = new_node();
        top->parent = c->parent;
        top->key.assign(c->key.begin(), c->key.begin() + k);
        top->slots.assign(c->slots.begin(), c->slots.begin() + k);
        top->stamp = c->stamp;
        top->ref = c->ref;
        top->depth = c->depth - (int64_t)(c->key.size() - k);
        c->key.erase(c->key.begin(), c->key.begin() + k);
        c->slots.erase(c->slots.begin(), c->slots.begin() + k);
        c->parent->children.set(top->key[0], top);
        add_child(top, c->key[0], c);
        c->parent = top;
        return top;
    }

    // Walk the cached path of tokens[0:n]: split where it ends inside an edge, stamp every
    // node on it, optionally collect slots.  Returns the matched length; *last = end node.
    int64_t walk(const int32_t* tokens, int64_t n, int32_t* out_slots, rx::Node** last) {
        return walk_from(&root, 0, tokens, n, out_slots, last);
    }

    // Length of the cached prefix of tokens[0:n], touching nothing.
    int64_t cached_len(const int32_t* tokens, int64_t n) const {
        const rx::Node* x = &root;
        int64_t pos = 0;
        while (pos < n) {
            const rx::Node* c = x->children.find(tokens[pos]);
            if (!c) break;
            const int64_t len = (int64_t)c->key.size();
            const int64_t k = rx::common_prefix(c->key.data(), tokens + pos, 1, std::min<int64_t>(len, n - pos));
            pos += k;
            if (k < len) break;
            x = c;
        }
        return pos;
    }

    // A request's reusable prefix: the cached prefix, cut down to whole pages when the page
    // size is above one (the walk then ends, splits and stamps at that page boundary).
    int64_t match(const int32_t* tokens, int64_t n, int32_t* out_slots, rx::Node** last) {
        if (page > 1) {
            const int64_t m = cached_len(tokens, n);
            n = m - m % page;
        }
        return walk(tokens, n, out_slots, last);
    }

    // The walk along a path already known to be cached for its first m tokens (a cached_len
    // result; splits since then move node boundaries, never what is cached): split where it
    // ends inside an edge and stamp every node on it, without comparing tokens again.
    // Returns the end node, or nullptr if the path is not there.
    rx::Node* walk_known(const int32_t* tokens, int64_t m) {
        rx::Node* x = &root;
        int64_t pos = 0;
        while (pos < m) {
            rx::Node* c = x->children.find(tokens[pos]);
            if (!c) return nullptr;
            const size_t len = c->key.size();
            const int64_t k = std::min<int64_t>((int64_t)len, m - pos);
            if ((size_t)k < len) c = split(c, (size_t)k);
            c->stamp = clock;
            pos += k;
            x = c;
        }
        return x;
    }

    // The slots of the whole root path ending at node x (which ends at depth x->depth).
    static void path_slots(const rx::Node* x, int32_t* out) {
        for (; x->parent != nullptr; x = x->parent) {
            const int64_t k = (int64_t)x->key.size();
            std::memcpy(out + (x->depth - k), x->slots.data(), sizeof(int32_t) * (size_t)k);
        }
    }

    // The walk continued from node x, which ends at token position pos of the sequence.
    int64_t walk_from(rx::Node* x, int64_t pos, const int32_t* tokens, int64_t n, int32_t* out_slots,
                      rx::Node** last) {
        while (pos < n) {
            rx::Node* c = x->children.find(tokens[pos]);
            if (!c) break;
            const size_t len = c->key.size();
            const int64_t lim = std::min<int64_t>((int64_t)len, n - pos);
            const int64_t k = rx::common_prefix(c->key.data(), tokens + pos, 1, lim);
            if ((size_t)k < len) c = split(c, (size_t)k);
            c->stamp = clock;
            if (out_slots) std::memcpy(out_slots + pos, c->slots.data(), sizeof(int32_t) * (size_t)k);
            pos += k;
            x = c;
            if ((size_t)k < len) break;
        }
        *last = x;
        return pos;
    }
};

using rx::set_error;

extern "C" {

const char* rx_last_error(void) { return rx::g_last_error.c_str(); }

const char* rx_version(void) { return "radixattn 0.1 (sm_103a)"; }

int rx_set_tracing(int on) { return rx::g_trace.exchange(on ? 1 : 0); }

int radix_create(int64_t num_slots, uint64_t slot_perm_seed, rx_radix** out) {
    RX_REQUIRE(out != nullptr, "radix_create: out is NULL");
    RX_REQUIRE(num_slots >= 1 && num_slots <= INT32_MAX, "radix_create: num_slots %lld out of range",
               (long long)num_slots);
    rx_radix* t = new (std::nothrow) rx_radix();
    if (!t) {
        set_error("radix_create: out of host memory");
        return RX_ENOMEM;
    }
    try {
        t->num_slots = num_slots;
        std::vector<std::pair<uint64_t, int32_t>> keyed((size_t)num_slots);
        for (int64_t i = 0; i < num_slots; ++i)
            keyed[(size_t)i] = {rx::splitmix64_at(slot_perm_seed, (uint64_t)i + 1), (int32_t)i};
        std::sort(keyed.begin(), keyed.end());
        t->ring.resize((size_t)num_slots);
        for (int64_t i = 0; i < num_slots; ++i) t->ring[(size_t)i] = keyed[(size_t)i].second;
        t->count = num_slots;
        t->is_free.assign((size_t)num_slots, 1);
    } catch (const std::bad_alloc&) {
        delete t;
        set_error("radix_create: out of host memory");
        return RX_ENOMEM;
    }
    t->root.id = 0;
    t->by_id.set(0, &t->root);
    t->st.num_slots = num_slots;
    *out = t;
    return RX_OK;
}

void radix_destroy(rx_radix* t) { delete t; }

int match_prefix(rx_radix* t, const int32_t* tokens, int64_t n, int32_t* out_slots, int64_t* out_len,
                 rx_node* out_last) {
    RX_TRACE("match_prefix");
    RX_REQUIRE(t && out_len && out_last && n >= 0 && (n == 0 || (tokens && out_slots)),
               "match_prefix: bad arguments");
    t->clock += 1;
    rx::Node* last = nullptr;
    const int64_t m = t->match(tokens, n, out_slots, &last);
    t->st.match_calls += 1;
    t->st.match_query_tokens += n;
    t->st.match_hit_tokens += m;
    *out_len = m;
    *out_last = last->id;
    return RX_OK;
}

int match_prefix_len(const rx_radix* t, const int32_t* tokens, int64_t n, int64_t* out_len) {
    RX_TRACE("match_prefix_len");
    RX_REQUIRE(t && out_len && n >= 0 && (n == 0 || tokens), "match_prefix_len: bad arguments");
    const int64_t m = t->cached_len(tokens, n);
    *out_len = m - m % t->page;         // the length match_prefix would return now
    return RX_OK;
}

int radix_set_page_size(rx_radix* t, int64_t page_size) {
    RX_REQUIRE(t && page_size >= 1 && page_size <= (1 << 20), "radix_set_page_size: page size %lld out of range",
               (long long)page_size);
    t->page = page_size;
    return RX_OK;
}

int match_prefix_len_batch(const rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                           int64_t* out_len) {
    RX_TRACE("match_prefix_len_batch");
    RX_REQUIRE(t && batch >= 0 && tok_indptr && (batch == 0 || out_len), "match_prefix_len_batch: bad arguments");
    for (int32_t b = 0; b < batch; ++b)
        RX_REQUIRE(tok_indptr[b + 1] >= tok_indptr[b], "match_prefix_len_batch: request %d has a negative length", b);
    RX_REQUIRE(batch == 0 || tokens || tok_indptr[batch] == tok_indptr[0], "match_prefix_len_batch: tokens is NULL");
    auto one = [&](int64_t b) {
        const int64_t m = t->cached_len(tokens + tok_indptr[b], tok_indptr[b + 1] - tok_indptr[b]);
        out_len[b] = m - m % t->page;
    };
    if (batch > 0 && tok_indptr[batch] - tok_indptr[0] >= rx::kParallelTokens) rx::Pool::get().run(batch, one);
    else
        for (int32_t b = 0; b < batch; ++b) one(b);
    return RX_OK;
}

int radix_lock(rx_radix* t, rx_node node) {
    RX_TRACE("radix_lock");
    RX_REQUIRE(t, "radix_lock: tree is NULL");
    rx::Node* const at = t->by_id.find(node);
    RX_REQUIRE(at, "radix_lock: unknown node %lld", (long long)node);
    for (rx::Node* x = at; x != &t->root; x = x->parent) x->ref += 1;
    return RX_OK;
}

int radix_unlock(rx_radix* t, rx_node node) {
    RX_TRACE("radix_unlock");
    RX_REQUIRE(t, "radix_unlock: tree is NULL");
    rx::Node* const at = t->by_id.find(node);
    RX_REQUIRE(at, "radix_unlock: unknown node %lld", (long long)node);
    for (rx::Node* x = at; x != &t->root; x = x->parent)
        if (x->ref <= 0) {
            set_error("radix_unlock: node %lld is not locked", (long long)node);
            return RX_ELOCKED;
        }
    for (rx::Node* x = at; x != &t->root; x = x->parent) x->ref -= 1;
    return RX_OK;
}

int radix_lock_batch(rx_radix* t, const rx_node* nodes, int32_t n) {
    RX_TRACE("radix_lock_batch");
    RX_REQUIRE(t && n >= 0 && (n == 0 || nodes), "radix_lock_batch: bad arguments");
    for (int32_t i = 0; i < n; ++i)
        RX_REQUIRE(t->by_id.find(nodes[i]), "radix_lock_batch: unknown node %lld", (long long)nodes[i]);
    for (int32_t i = 0; i < n; ++i) radix_lock(t, nodes[i]);
    return RX_OK;
}

int radix_unlock_batch(rx_radix* t, const rx_node* nodes, int32_t n) {
    RX_TRACE("radix_unlock_batch");
    RX_REQUIRE(t && n >= 0 && (n == 0 || nodes), "radix_unlock_batch: bad arguments");
    for (int32_t i = 0; i < n; ++i) {
        const int rc = radix_unlock(t, nodes[i]);
        if (rc != RX_OK) return rc;
    }
    return RX_OK;
}

int alloc_slots(rx_radix* t, int64_t n, int32_t* out_slots) {
    RX_TRACE("alloc_slots");
    RX_REQUIRE(t && n >= 0 && (n == 0 || out_slots), "alloc_slots: bad arguments");
    if (n > t->count) {
        set_error("alloc_slots: %lld slots requested, %lld free", (long long)n, (long long)t->count);
        return RX_ENOMEM;
    }
    // at most two contiguous runs of the ring: from head to its end, then from its start
    if (n == 0) return RX_OK;
    const int64_t first = std::min<int64_t>(n, t->num_slots - t->head);
    std::memcpy(out_slots, t->ring.data() + t->head, sizeof(int32_t) * (size_t)first);
    if (n > first) std::memcpy(out_slots + first, t->ring.data(), sizeof(int32_t) * (size_t)(n - first));
    for (int64_t i = 0; i < n; ++i) t->is_free[(size_t)out_slots[i]] = 0;
    t->head = t->ring_pos(n);
    t->count -= n;
    return RX_OK;
}

int free_slots(rx_radix* t, const int32_t* slots, int64_t n) {
    RX_TRACE("free_slots");
    RX_REQUIRE(t && n >= 0 && (n == 0 || slots), "free_slots: bad arguments");
    int64_t i = 0;
    for (; i < n; ++i) {
        const int32_t s = slots[i];
        if (s < 0 || s >= t->num_slots || t->is_free[(size_t)s]) break;
        t->is_free[(size_t)s] = 1;   // mark now to catch repeats within the call
    }
    if (i < n) {
        const int32_t bad = slots[i];
        for (int64_t j = 0; j < i; ++j) t->is_free[(size_t)slots[j]] = 0;   // roll back
        set_error("free_slots: slot %d is out of range, already free or repeated", bad);
        return RX_EINVAL;
    }
    for (i = 0; i < n; ++i) {
        t->ring[(size_t)t->ring_pos(t->count)] = slots[i];
        t->count += 1;
    }
    return RX_OK;
}

int insert(rx_radix* t, const int32_t* tokens, const int32_t* slots, int64_t n, int64_t* out_dup_len,
           rx_node* out_last) {
    RX_TRACE("insert");
    RX_REQUIRE(t && out_dup_len && out_last && n >= 0 && (n == 0 || (tokens && slots)),
               "insert: bad arguments");
    // Validate the slots the tree would take before changing anything.
    {
        rx::Node* x = &t->root;
        int64_t pos = 0;   // non-mutating walk to find dup_len
        while (pos < n) {
            rx::Node* c = x->children.find(tokens[pos]);
            if (!c) break;
            const int64_t lim = std::min<int64_t>((int64_t)c->key.size(), n - pos);
            int64_t k = 1;
            while (k < lim && c->key[k] == tokens[pos + k]) ++k;
            pos += k;
            if (k < (int64_t)c->key.size()) break;
            x = c;
        }
        for (int64_t i = pos; i < n; ++i)
            RX_REQUIRE(slots[i] >= 0 && slots[i] < t->num_slots && !t->is_free[(size_t)slots[i]],
                       "insert: slot %d at position %lld is out of range or free", slots[i], (long long)i);
    }
    t->clock += 1;
    rx::Node* x = nullptr;
    const int64_t dup = t->walk(tokens, n, nullptr, &x);
    if (dup < n) {
        rx::Node* leaf = t->new_node();
        leaf->parent = x;
        leaf->key.assign(tokens + dup, tokens + n);
        leaf->slots.assign(slots + dup, slots + n);
        leaf->stamp = t->clock;
        leaf->depth = x->depth + (n - dup);
        t->add_child(x, tokens[dup], leaf);
        x = leaf;
        t->st.cached_tokens += n - dup;
        t->st.inserted_tokens += n - dup;
    }
    t->st.insert_calls += 1;
    *out_dup_len = dup;
    *out_last = x->id;
    return RX_OK;
}

int evict(rx_radix* t, int64_t num_tokens, int32_t* out_freed, int64_t cap, int64_t* out_n) {
    RX_TRACE("evict");
    RX_REQUIRE(t && out_n && num_tokens >= 0 && cap >= 0, "evict: bad arguments");
    if (num_tokens == 0) {
        *out_n = 0;
        return RX_OK;
    }
    // Collect the evictable leaves into a min-heap on (stamp, id).
    auto& heap = t->ev_heap;
    auto& stack = t->ev_stack;
    const std::greater<rx_radix::EvictItem> later;
    heap.clear();
    stack.clear();
    stack.push_back(&t->root);
    while (!stack.empty()) {
        rx::Node* x = stack.back();
        stack.pop_back();
        if (x != &t->root && x->children.empty() && x->ref == 0) heap.emplace_back(x->stamp, x->id, x);
        x->children.for_each([&](int32_t, rx::Node* c) { stack.push_back(c); });
    }
    std::make_heap(heap.begin(), heap.end(), later);
    int64_t freed = 0;
    while (freed < num_tokens && !heap.empty()) {
        std::pop_heap(heap.begin(), heap.end(), later);
        rx::Node* x = std::get<2>(heap.back());
        heap.pop_back();
        for (int32_t s : x->slots) {
            if (out_freed && freed < cap) out_freed[freed] = s;
            t->push_free(s);
            ++freed;
        }
        rx::Node* p = x->parent;
        t->drop_child(p, x->key[0]);
        t->st.cached_tokens -= (int64_t)x->key.size();
        t->drop_id(x->id);
        --t->st.node_count;
        if (t->spare.size() < rx_radix::kSpareNodes) t->spare.push_back(x);
        else delete x;
        if (p != &t->root && p->children.empty() && p->ref == 0) {
            heap.emplace_back(p->stamp, p->id, p);
            std::push_heap(heap.begin(), heap.end(), later);
        }
    }
    t->st.evicted_tokens += freed;
    *out_n = freed;
    return RX_OK;
}

int match_prefix_batch(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                       int32_t* out_slots, int64_t* out_indptr, rx_node* out_last) {
    RX_TRACE("match_prefix_batch");
    RX_REQUIRE(t && batch >= 0 && tok_indptr && out_indptr && (batch == 0 || out_last),
               "match_prefix_batch: bad arguments");
    out_indptr[0] = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t n = tok_indptr[b + 1] - tok_indptr[b];
        RX_REQUIRE(n >= 0 && tok_indptr[b] >= 0, "match_prefix_batch: bad tok_indptr at %d", b);
        int64_t len = 0;
        const int rc = match_prefix(t, tokens + tok_indptr[b], n, out_slots + out_indptr[b], &len, out_last + b);
        if (rc != RX_OK) return rc;
        out_indptr[b + 1] = out_indptr[b] + len;
    }
    return RX_OK;
}

int insert_batch(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                 const int32_t* slots, int64_t* out_dup_len, rx_node* out_last) {
    RX_TRACE("insert_batch");
    RX_REQUIRE(t && batch >= 0 && tok_indptr && (batch == 0 || (out_dup_len && out_last)),
               "insert_batch: bad arguments");
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t n = tok_indptr[b + 1] - tok_indptr[b];
        RX_REQUIRE(n >= 0 && tok_indptr[b] >= 0, "insert_batch: bad tok_indptr at %d", b);
        const int rc = insert(t, tokens + tok_indptr[b], slots + tok_indptr[b], n, out_dup_len + b, out_last + b);
        if (rc != RX_OK) return rc;
    }
    return RX_OK;
}

int insert_batch_at(rx_radix* t, int32_t batch, const rx_node* nodes, const int32_t* tokens,
                    const int64_t* tok_indptr, const int32_t* new_slots, const int64_t* new_indptr,
                    int64_t* out_dup_len, rx_node* out_last) {
    RX_TRACE("insert_batch_at");
    RX_REQUIRE(t && batch >= 0 && (batch == 0 || (nodes && tokens && tok_indptr && new_indptr && out_dup_len && out_last)),
               "insert_batch_at: bad arguments");
    for (int32_t b = 0; b < batch; ++b) {
        rx::Node* x = t->by_id.find(nodes[b]);
        RX_REQUIRE(x, "insert_batch_at: unknown node %lld", (long long)nodes[b]);
        const int64_t n = tok_indptr[b + 1] - tok_indptr[b];
        const int64_t d = x->depth;
        const int64_t m = new_indptr[b + 1] - new_indptr[b];
        RX_REQUIRE(d >= 0 && d <= n && m == n - d, "insert_batch_at: request %d: node depth %lld, %lld tokens, %lld new slots",
                   b, (long long)d, (long long)n, (long long)m);
        const int32_t* tok = tokens + tok_indptr[b];
        const int32_t* sl = new_slots + new_indptr[b];
        for (int64_t i = 0; i < m; ++i)
            RX_REQUIRE(sl[i] >= 0 && sl[i] < t->num_slots && !t->is_free[(size_t)sl[i]],
                       "insert_batch_at: slot %d of request %d is out of range or free", sl[i], b);
        t->clock += 1;
        for (rx::Node* y = x; y != &t->root; y = y->parent) y->stamp = t->clock;   // the cached path
        rx::Node* end = nullptr;
        const int64_t dup = t->walk_from(x, d, tok, n, nullptr, &end);
        if (dup < n) {
            rx::Node* leaf = t->new_node();
            leaf->parent = end;
            leaf->key.assign(tok + dup, tok + n);
            leaf->slots.assign(sl + (dup - d), sl + m);
            leaf->stamp = t->clock;
            leaf->depth = end->depth + (n - dup);
            t->add_child(end, tok[dup], leaf);
            end = leaf;
            t->st.cached_tokens += n - dup;
            t->st.inserted_tokens += n - dup;
        }
        t->st.insert_calls += 1;
        out_dup_len[b] = dup;
        out_last[b] = end->id;
    }
    return RX_OK;
}

static inline int64_t up256(int64_t x) { return (x + 255) & ~(int64_t)255; }

size_t rx_step_stage_bytes(int32_t batch, int64_t total_tokens) {
    if (batch < 0 || total_tokens < 0) return 0;
    const int64_t b1 = (int64_t)batch + 1;
    return (size_t)(up256(4 * total_tokens) + up256(8 * b1) + up256(4 * total_tokens) + up256(8 * b1) +
                    up256(4 * (int64_t)batch) + up256(4 * (int64_t)batch) + up256(4 * b1) + up256(4 * (int64_t)batch) +
                    up256(4 * (int64_t)batch) + 256);
}

int rx_step_plan(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr, const int32_t* n_new,
                 int32_t group_mode, int32_t heads_per_kv, int64_t min_shared, void* h_stage, size_t stage_cap,
                 rx_node* out_last, rx_step_layout* out) {
    RX_TRACE("rx_step_plan");
    RX_REQUIRE(t && batch >= 0 && tok_indptr && out && h_stage && (batch == 0 || (tokens && n_new && out_last)),
               "rx_step_plan: bad arguments");
    const int64_t total_tokens = tok_indptr[batch];
    RX_REQUIRE(stage_cap >= rx_step_stage_bytes(batch, total_tokens), "rx_step_plan: staging buffer of %zu bytes, %zu needed",
               stage_cap, rx_step_stage_bytes(batch, total_tokens));
    unsigned char* st = (unsigned char*)h_stage;
    rx_step_layout L{};
    L.batch = batch;
    // a1: matched slots straight into the staging buffer
    L.off_prefix_slots = 0;
    int32_t* ps = (int32_t*)(st + L.off_prefix_slots);
    std::vector<int64_t> P((size_t)batch);
    int64_t acc = 0, T = 0;
    int32_t max_qo = 0, max_kv = 1;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t len = tok_indptr[b + 1] - tok_indptr[b];
        RX_REQUIRE(len >= 0 && n_new[b] >= 0 && n_new[b] <= len, "rx_step_plan: request %d: %lld tokens, %d new", b,
                   (long long)len, n_new[b]);
    }
    // Every prompt is read against the tree first (in parallel: the reads are independent and
    // nothing changes the tree meanwhile); the match lengths are checked before anything is
    // stamped, split or allocated.
    const bool par = batch > 0 && total_tokens - tok_indptr[0] >= rx::kParallelTokens;
    {
        auto one = [&](int64_t b) {
            const int64_t m = t->cached_len(tokens + tok_indptr[b], tok_indptr[b + 1] - tok_indptr[b]);
            P[(size_t)b] = m - m % t->page;
        };
        if (par) rx::Pool::get().run(batch, one);
        else
            for (int32_t b = 0; b < batch; ++b) one(b);
    }
    std::vector<int64_t> off((size_t)batch + 1, 0);
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t len = tok_indptr[b + 1] - tok_indptr[b];
        RX_REQUIRE(P[(size_t)b] + n_new[b] == len, "rx_step_plan: request %d: %lld tokens cached, %lld expected", b,
                   (long long)P[(size_t)b], (long long)(len - n_new[b]));
        off[(size_t)b + 1] = off[(size_t)b] + P[(size_t)b];
    }
    // Then, in request order, each walk splits at its match end and stamps its path (one
    // clock tick per request), without comparing tokens again.
    std::vector<rx::Node*> lastn((size_t)batch);
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t len = tok_indptr[b + 1] - tok_indptr[b];
        t->clock += 1;
        rx::Node* last = t->walk_known(tokens + tok_indptr[b], P[(size_t)b]);
        RX_REQUIRE(last != nullptr, "rx_step_plan: request %d: cached path changed during the plan", b);
        lastn[(size_t)b] = last;
        t->st.match_calls += 1;
        t->st.match_query_tokens += len;
        t->st.match_hit_tokens += P[(size_t)b];
        out_last[b] = last->id;
        acc += P[(size_t)b];
        T += n_new[b];
        max_qo = std::max(max_qo, n_new[b]);
        max_kv = std::max<int32_t>(max_kv, (int32_t)len);
    }
    // The matched slots, copied along each final path (in parallel: no split happens now).
    {
        auto one = [&](int64_t b) { rx_radix::path_slots(lastn[(size_t)b], ps + off[(size_t)b]); };
        if (par) rx::Pool::get().run(batch, one);
        else
            for (int32_t b = 0; b < batch; ++b) one(b);
    }
    L.total_prefix = acc;
    L.total_new = T;
    L.max_qo_len = max_qo;
    L.max_kv_len = max_kv;
    L.stride = (max_kv + 7) / 8 * 8;
    L.off_prefix_indptr = up256(4 * acc);
    L.off_new_slots = L.off_prefix_indptr + up256(8 * ((int64_t)batch + 1));
    L.off_qo_indptr = L.off_new_slots + up256(4 * T);
    L.off_prefix_lens = L.off_qo_indptr + up256(8 * ((int64_t)batch + 1));
    L.off_kv_lens = L.off_prefix_lens + up256(4 * (int64_t)batch);
    L.off_grp_indptr = L.off_kv_lens + up256(4 * (int64_t)batch);
    L.off_grp_members = L.off_grp_indptr + up256(4 * ((int64_t)batch + 1));
    L.off_grp_len = L.off_grp_members + up256(4 * (int64_t)batch);
    L.bytes = L.off_kv_lens + up256(4 * (int64_t)batch);
    // a2: allocate the new tokens' slots
    int32_t* ns = (int32_t*)(st + L.off_new_slots);
    {
        const int rc = alloc_slots(t, T, ns);
        if (rc != RX_OK) return rc;
    }
    int64_t* pind = (int64_t*)(st + L.off_prefix_indptr);
    int64_t* qo = (int64_t*)(st + L.off_qo_indptr);
    int32_t* pl = (int32_t*)(st + L.off_prefix_lens);
    int32_t* kl = (int32_t*)(st + L.off_kv_lens);
    pind[0] = 0;
    qo[0] = 0;
    for (int32_t b = 0; b < batch; ++b) {
        pind[b + 1] = pind[b] + P[(size_t)b];
        qo[b + 1] = qo[b] + n_new[b];
        pl[b] = (int32_t)P[(size_t)b];
        kl[b] = (int32_t)(P[(size_t)b] + n_new[b]);
    }
    // optional shared-prefix groups ("auto": not for the small-extend shape -- a few rows per
    // (request, kv head) over at most 1024 keys -- which needs no stacking)
    const bool small_shape = (int64_t)max_qo * heads_per_kv <= 8 && max_kv <= 1024;
    bool want_groups = group_mode != RX_GROUPS_NONE && batch > 0 && !(group_mode == RX_GROUPS_AUTO && small_shape);
    // "auto" never stacks a request with 128 or more new rows per kv head: decided from n_new
    // alone, before the groups are derived from the tree (which would be discarded)
    if (want_groups && group_mode == RX_GROUPS_AUTO)
        for (int32_t b = 0; b < batch && want_groups; ++b)
            if ((int64_t)n_new[b] * heads_per_kv >= 128) want_groups = false;
    if (want_groups) {
        std::vector<int32_t> gof((size_t)batch);
        std::vector<int64_t> glen((size_t)batch);
        int32_t ng = 0;
        int rc = radix_shared_groups(t, out_last, batch, min_shared, gof.data(), glen.data(), &ng);
        if (rc != RX_OK) {
            free_slots(t, ns, T);
            return rc;
        }
        bool use = ng > 0;
        if (use && group_mode == RX_GROUPS_AUTO) {
            for (int32_t b = 0; b < batch && use; ++b) {
                if (gof[(size_t)b] < 0) use = false;
                else if (P[(size_t)b] + n_new[b] - glen[(size_t)gof[(size_t)b]] > 256) use = false;
                else if ((int64_t)n_new[b] * heads_per_kv >= 128) use = false;
            }
        }
        if (use) {
            int32_t* gi = (int32_t*)(st + L.off_grp_indptr);
            int32_t* gm = (int32_t*)(st + L.off_grp_members);
            int32_t* gl = (int32_t*)(st + L.off_grp_len);
            std::vector<int32_t> cnt((size_t)ng, 0);
            std::vector<int64_t> rows((size_t)ng, 0);
            for (int32_t b = 0; b < batch; ++b)
                if (gof[(size_t)b] >= 0) {
                    cnt[(size_t)gof[(size_t)b]] += 1;
                    rows[(size_t)gof[(size_t)b]] += n_new[b];
                }
            gi[0] = 0;
            for (int32_t g = 0; g < ng; ++g) gi[g + 1] = gi[g] + cnt[(size_t)g];
            std::vector<int32_t> fill(gi, gi + ng);
            for (int32_t b = 0; b < batch; ++b)
                if (gof[(size_t)b] >= 0) gm[fill[(size_t)gof[(size_t)b]]++] = b;
            for (int32_t g = 0; g < ng; ++g) {
                gl[g] = (int32_t)glen[(size_t)g];
                L.max_group_size = std::max(L.max_group_size, cnt[(size_t)g]);
                L.max_group_len = std::max(L.max_group_len, gl[g]);
                L.max_group_rows = std::max<int32_t>(L.max_group_rows, (int32_t)rows[(size_t)g]);
            }
            L.num_groups = ng;
            L.bytes = L.off_grp_len + up256(4 * (int64_t)ng);
        }
    }
    // pin the matched prefixes for the step (last, so that a failure above leaves none pinned)
    for (int32_t b = 0; b < batch; ++b)
        for (rx::Node* x = t->by_id.find(out_last[b]); x != &t->root; x = x->parent) x->ref += 1;
    *out = L;
    return RX_OK;
}

int rx_step_finish(rx_radix* t, int32_t batch, const int32_t* tokens, const int64_t* tok_indptr,
                   const rx_node* last_nodes, const void* h_stage, const rx_step_layout* L, int64_t evict_tokens,
                   int64_t* out_evicted) {
    RX_TRACE("rx_step_finish");
    RX_REQUIRE(t && L && h_stage && batch == L->batch && (batch == 0 || (tokens && tok_indptr && last_nodes)),
               "rx_step_finish: bad arguments");
    const unsigned char* st = (const unsigned char*)h_stage;
    const int32_t* ns = (const int32_t*)(st + L->off_new_slots);
    const int64_t* qo = (const int64_t*)(st + L->off_qo_indptr);
    const int32_t* pl = (const int32_t*)(st + L->off_prefix_lens);
    std::vector<int64_t> dup((size_t)std::max(batch, 1));
    std::vector<rx_node> last((size_t)std::max(batch, 1));
    int rc = insert_batch_at(t, batch, last_nodes, tokens, tok_indptr, ns, qo, dup.data(), last.data());
    if (rc != RX_OK) return rc;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t over = dup[(size_t)b] - pl[b];   // new slots whose tokens were cached meanwhile
        if (over > 0) {
            rc = free_slots(t, ns + qo[b], over);
            if (rc != RX_OK) return rc;
        }
    }
    int64_t freed = 0;
    if (evict_tokens > 0) {
        rc = evict(t, evict_tokens, nullptr, 0, &freed);
        if (rc != RX_OK) return rc;
    }
    if (out_evicted) *out_evicted = freed;
    return radix_unlock_batch(t, last_nodes, batch);
}

int radix_stats(const rx_radix* t, rx_stats* out) {
    RX_REQUIRE(t && out, "radix_stats: bad arguments");
    *out = t->st;
    out->free_slots = t->count;
    out->num_slots = t->num_slots;
    return RX_OK;
}

int radix_check(const rx_radix* t) {
    RX_TRACE("radix_check");
    RX_REQUIRE(t, "radix_check: tree is NULL");
    std::vector<uint8_t> owned((size_t)t->num_slots, 0);
    int64_t nodes = 0, tokens = 0;
    std::vector<const rx::Node*> stack{&t->root};
    while (!stack.empty()) {
        const rx::Node* x = stack.back();
        stack.pop_back();
        int64_t child_ref = 0;
        std::vector<std::pair<int32_t, const rx::Node*>> kids;
        x->children.for_each([&](int32_t tok, const rx::Node* c) { kids.emplace_back(tok, c); });
        for (const auto& kv : kids) {
            const rx::Node* c = kv.second;
            RX_REQUIRE(c->parent == x, "radix_check: node %lld has a wrong parent", (long long)c->id);
            RX_REQUIRE(!c->key.empty() && c->key.size() == c->slots.size(),
                       "radix_check: node %lld has an empty or unbalanced edge", (long long)c->id);
            RX_REQUIRE(c->key[0] == kv.first, "radix_check: node %lld is filed under a wrong token",
                       (long long)c->id);
            RX_REQUIRE(c->depth == x->depth + (int64_t)c->key.size(), "radix_check: node %lld depth",
                       (long long)c->id);
            RX_REQUIRE(x == &t->root || c->stamp <= x->stamp,
                       "radix_check: node %lld is more recent than its parent", (long long)c->id);
            RX_REQUIRE(c->ref >= 0, "radix_check: node %lld has a negative lock count", (long long)c->id);
            RX_REQUIRE(t->by_id.find(c->id) == c, "radix_check: handle of node %lld", (long long)c->id);
            child_ref += c->ref;
            stack.push_back(c);
        }
        RX_REQUIRE(x == &t->root || x->ref >= child_ref, "radix_check: node %lld holds fewer locks than its children",
                   (long long)x->id);
        if (x != &t->root) {
            ++nodes;
            tokens += (int64_t)x->key.size();
            for (int32_t s : x->slots) {
                RX_REQUIRE(s >= 0 && s < t->num_slots, "radix_check: slot %d out of range", s);
                RX_REQUIRE(!owned[(size_t)s], "radix_check: slot %d held twice", s);
                RX_REQUIRE(!t->is_free[(size_t)s], "radix_check: slot %d is cached and free", s);
                owned[(size_t)s] = 1;
            }
        }
    }
    RX_REQUIRE(nodes == t->st.node_count && (int64_t)t->by_id.size() == nodes + 1,
               "radix_check: node count %lld vs %lld", (long long)nodes, (long long)t->st.node_count);
    RX_REQUIRE(tokens == t->st.cached_tokens, "radix_check: cached tokens %lld vs %lld", (long long)tokens,
               (long long)t->st.cached_tokens);
    int64_t nfree = 0;
    for (uint8_t f : t->is_free) nfree += f;
    RX_REQUIRE(nfree == t->count, "radix_check: free bitmap %lld vs ring %lld", (long long)nfree,
               (long long)t->count);
    for (int64_t i = 0; i < t->count; ++i) {
        const int32_t s = t->ring[(size_t)((t->head + i) % t->num_slots)];
        RX_REQUIRE(t->is_free[(size_t)s], "radix_check: ring holds a used slot %d", s);
    }
    return RX_OK;
}

int radix_shared_groups(const rx_radix* t, const rx_node* last_nodes, int32_t batch, int64_t min_shared,
                        int32_t* out_group_of, int64_t* out_group_len, int32_t* out_num_groups) {
    RX_TRACE("radix_shared_groups");
    RX_REQUIRE(t && batch >= 0 && out_num_groups && (batch == 0 || (last_nodes && out_group_of && out_group_len)),
               "radix_shared_groups: bad arguments");
    // Root paths of every request's end node (root excluded), shallow to deep.
    std::vector<std::vector<const rx::Node*>> paths((size_t)batch);
    for (int32_t b = 0; b < batch; ++b) {
        const rx::Node* const at = t->by_id.find(last_nodes[b]);
        RX_REQUIRE(at, "radix_shared_groups: unknown node %lld", (long long)last_nodes[b]);
        for (const rx::Node* x = at; x != &t->root; x = x->parent) paths[(size_t)b].push_back(x);
        std::reverse(paths[(size_t)b].begin(), paths[(size_t)b].end());
    }
    std::unordered_map<const rx::Node*, std::vector<int32_t>> by_top;
    std::vector<const rx::Node*> order;
    for (int32_t b = 0; b < batch; ++b) {
        out_group_of[b] = -1;
        if (paths[(size_t)b].empty()) continue;
        const rx::Node* top = paths[(size_t)b][0];
        auto& v = by_top[top];
        if (v.empty()) order.push_back(top);
        v.push_back(b);
    }
    int32_t ng = 0;
    for (const rx::Node* top : order) {
        const auto& mem = by_top[top];
        if (mem.size() < 2) continue;
        size_t common = paths[(size_t)mem[0]].size();
        for (int32_t b : mem) {
            const auto& p = paths[(size_t)b];
            size_t i = 0;
            while (i < common && i < p.size() && p[i] == paths[(size_t)mem[0]][i]) ++i;
            common = i;
        }
        const int64_t len = paths[(size_t)mem[0]][common - 1]->depth;
        if (len < min_shared) continue;
        for (int32_t b : mem) out_group_of[b] = ng;
        out_group_len[ng] = len;
        ++ng;
    }
    *out_num_groups = ng;
    return RX_OK;
}

}  // extern "C"
