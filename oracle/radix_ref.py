"""Oracle for the radix prefix cache (test infrastructure only).

A deliberately naive model of the prefix cache that shares nothing with the C++ tree:

* ``ListMatcher`` -- the list-based matcher: a list of stored (tokens, slots) records;
  a lookup returns the longest common prefix over all records and that record's slots.
* ``PrefixCacheModel`` -- the cache kept as a dictionary from every cached token PREFIX
  (a tuple) to its slot, LRU stamp and lock count, plus the set of prefixes at which a
  node boundary was cut.  Nodes are never materialised: a node is the maximal run of
  cached positions between boundaries, computed on demand.  This reproduces the node
  structure, LRU order and eviction of a radix tree without building one.
* ``SlotAllocator`` -- the seeded free list, replayed from the published SplitMix64
  output function.
* ``req_to_token`` -- the per-request slot table: matched slots followed by new slots.

What it follows:
 - "SGLang: Efficient Execution of Structured Language Model Programs" (unite.ai),
   RadixAttention bullet of the introduction: the runtime keeps an LRU cache of KV cache
   in a radix tree and uses the tree for matching, insertion and eviction.
 - Same page, the nine-step walk-through of the radix tree under an LRU policy: a new
   turn is inserted as a node; a prompt whose prefix is cached reuses that KV; a node is
   split in two when a new sequence shares only part of it; under memory pressure the
   least recently used nodes are evicted.
 - "Prompt Caching" (Ultralytics glossary), "How prompt caching works": the cache is
   reused only for an exactly matching prefix.

Readings where the pages leave the step open (each also listed in the design notes):
 - Token granularity: every cached token has its own slot.
 - A node boundary is cut at every divergence point and at the end of every match and
   every insert; nodes never merge again (evicting one branch of a divergence point leaves
   the boundary in place).  So a call stamps whole nodes.
 - LRU clock: +1 per match or insert call; every cached position on the touched path
   gets the new stamp.  Leaves are evicted whole, least recent stamp first; locked
   positions (and, through the lock path, their ancestors) are never evicted.
 - Insert over a cached prefix keeps the cached slots and reports how many leading
   positions were already present (``dup_len``); the caller owns slots[:dup_len].
 - Free list is FIFO: allocation pops from the head, frees append to the tail; the
   initial order is the slot ids sorted by their SplitMix64 output (ties by id).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1


# --------------------------------------------------------------------------- SplitMix64
def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """SplitMix64 output for the 1-based counters (Steele, Lea & Flood, OOPSLA 2014;
    the widely published splitmix64.c): state = seed + i * 0x9E3779B97F4A7C15, then the
    mix z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
    z ^= z >> 31.  numpy uint64 arithmetic wraps modulo 2**64 as the definition needs."""
    i = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & MASK64) + i * np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def slot_order(num_slots: int, seed: int) -> np.ndarray:
    """Initial free-list order: slot ids sorted by SplitMix64(seed, id + 1), ties by id."""
    keys = splitmix64(seed, np.arange(1, num_slots + 1, dtype=np.uint64))
    return np.argsort(keys, kind="stable").astype(np.int32)


class SlotAllocator:
    """FIFO free list of KV-pool slots."""

    def __init__(self, num_slots: int, seed: int):
        self.num_slots = num_slots
        self.free = list(slot_order(num_slots, seed).tolist())
        self.is_free = np.ones(num_slots, bool)

    def alloc(self, n: int):
        if n > len(self.free):
            return None
        out, self.free = self.free[:n], self.free[n:]
        self.is_free[out] = False
        return np.array(out, np.int32)

    def release(self, slots) -> bool:
        slots = [int(s) for s in slots]
        if any(s < 0 or s >= self.num_slots or self.is_free[s] for s in slots) or len(set(slots)) != len(slots):
            return False
        self.free.extend(slots)
        self.is_free[slots] = True
        return True


# --------------------------------------------------------------------------- list matcher
class ListMatcher:
    """Naive longest-prefix matcher over a list of stored (tokens, slots) records."""

    def __init__(self):
        self.records = []

    def add(self, tokens, slots):
        self.records.append((np.asarray(tokens, np.int32).copy(), np.asarray(slots, np.int32).copy()))

    def match(self, tokens):
        tokens = np.asarray(tokens, np.int32)
        best_len, best_slots = 0, np.zeros(0, np.int32)
        for rt, rs in self.records:
            n = min(len(rt), len(tokens))
            neq = np.flatnonzero(rt[:n] != tokens[:n])
            lcp = int(neq[0]) if len(neq) else n
            if lcp > best_len:
                best_len, best_slots = lcp, rs[:lcp]
        return best_len, best_slots.copy()


# --------------------------------------------------------------------------- prefix model
class PrefixCacheModel:
    """Radix prefix cache modelled as a dictionary of cached token prefixes."""

    def __init__(self, num_slots: int, seed: int):
        self.alloc = SlotAllocator(num_slots, seed)
        self.entries = {}        # prefix tuple -> [slot, stamp, ref]
        self.nchild = {(): 0}    # prefix tuple -> number of cached one-token extensions
        self.cuts = set()        # prefixes after which a node boundary was cut
        self.clock = 0
        self.stats = dict(match_calls=0, match_query_tokens=0, match_hit_tokens=0,
                          insert_calls=0, inserted_tokens=0, evicted_tokens=0)

    # ---- structure helpers
    def _cached_len(self, tokens) -> int:
        n = 0
        while n < len(tokens) and tuple(tokens[: n + 1]) in self.entries:
            n += 1
        return n

    def _is_boundary(self, p: tuple) -> bool:
        return p == () or p in self.cuts or self.nchild.get(p, 0) != 1

    def node_of(self, p: tuple):
        """Positions (as prefixes, shallow to deep) of the node containing cached prefix p."""
        start = p
        while len(start) > 1 and not self._is_boundary(start[:-1]):
            start = start[:-1]
        end = p
        while not self._is_boundary(end):
            (child,) = [c for c in self._children(end)]
            end = child
        return [end[:i] for i in range(len(start), len(end) + 1)]

    def _children(self, p: tuple):
        return [e for e in self.entries if len(e) == len(p) + 1 and e[:-1] == p]

    def nodes(self):
        """Every node as the list of its positions; node ends are the boundary positions."""
        return [self.node_of(p) for p in self.entries if self._is_boundary(p)]

    def _stamp(self, tokens, n):
        for i in range(n):
            self.entries[tuple(tokens[: i + 1])][1] = self.clock

    # ---- operations
    def match(self, tokens):
        tokens = [int(t) for t in tokens]
        self.clock += 1
        m = self._cached_len(tokens)
        self._stamp(tokens, m)
        if m > 0:
            self.cuts.add(tuple(tokens[:m]))
        self.stats["match_calls"] += 1
        self.stats["match_query_tokens"] += len(tokens)
        self.stats["match_hit_tokens"] += m
        return m, np.array([self.entries[tuple(tokens[: i + 1])][0] for i in range(m)], np.int32)

    def insert(self, tokens, slots):
        tokens = [int(t) for t in tokens]
        slots = [int(s) for s in slots]
        self.clock += 1
        dup = self._cached_len(tokens)
        if 0 < dup < len(tokens):
            self.cuts.add(tuple(tokens[:dup]))   # divergence point: a permanent boundary
        for i in range(dup, len(tokens)):
            p = tuple(tokens[: i + 1])
            self.entries[p] = [slots[i], 0, 0]
            self.nchild[p] = 0
            self.nchild[p[:-1]] = self.nchild.get(p[:-1], 0) + 1
        self._stamp(tokens, len(tokens))
        if tokens:
            self.cuts.add(tuple(tokens))
        self.stats["insert_calls"] += 1
        self.stats["inserted_tokens"] += len(tokens) - dup
        return dup

    def lock(self, tokens, n, delta=1):
        """Lock (delta=+1) or unlock (-1) the cached path tokens[:n]."""
        for i in range(n):
            self.entries[tuple(tokens[: i + 1])][2] += delta

    def evict(self, k: int):
        """Free unlocked least-recently-used leaf nodes until >= k tokens are freed."""
        freed = []
        while len(freed) < k:
            cands = []
            for p in self.entries:
                if self.nchild[p] == 0:          # deepest position of a leaf node
                    node = self.node_of(p)
                    if all(self.entries[x][2] == 0 for x in node):
                        cands.append((self.entries[p][1], node))
            if not cands:
                break
            stamp, node = min(cands, key=lambda c: c[0])
            for x in node:                       # shallow to deep: slots in position order
                freed.append(self.entries[x][0])
            for x in reversed(node):
                del self.entries[x]
                del self.nchild[x]
                self.nchild[x[:-1]] -= 1
                self.cuts.discard(x)
        self.alloc.release(freed)
        self.stats["evicted_tokens"] += len(freed)
        return np.array(freed, np.int32)

    def cached_tokens(self) -> int:
        return len(self.entries)

    def check_stamps_uniform(self) -> bool:
        """Every node's positions carry one stamp (the reading that calls stamp whole nodes)."""
        return all(len({self.entries[x][1] for x in node}) == 1 for node in self.nodes())


# --------------------------------------------------------------------------- shared groups
def shared_groups(matched, min_shared: int = 1):
    """Requests whose cached prefixes share their first node, and how long the common part is.

    matched: each request's matched (cached) token prefix.  Requests with a non-empty match
    are grouped by its first token (the root's child they go through), groups in order of
    first appearance; a group of two or more whose members' longest common prefix is at
    least min_shared keeps that length, the others are dropped (-1).  This is the reading
    behind reading a shared prefix once per group (the "SGLang" page's shared-prefix reuse
    across requests): the common prefix of cached paths ends at a node boundary, since a
    divergence point is always cut."""
    first, order = {}, []
    for b, p in enumerate(matched):
        if len(p) == 0:
            continue
        key = int(p[0])
        if key not in first:
            first[key] = []
            order.append(key)
        first[key].append(b)
    group_of, lens = [-1] * len(matched), []
    for key in order:
        mem = first[key]
        if len(mem) < 2:
            continue
        a = [int(t) for t in matched[mem[0]]]
        lcp = len(a)
        for b in mem[1:]:
            o = [int(t) for t in matched[b]]
            n = 0
            while n < min(lcp, len(o)) and o[n] == a[n]:
                n += 1
            lcp = n
        if lcp < min_shared:
            continue
        for b in mem:
            group_of[b] = len(lens)
        lens.append(lcp)
    return np.array(group_of, np.int32), np.array(lens, np.int64)


# --------------------------------------------------------------------------- slot table
def req_to_token(prefix_slots, new_slots, stride: int) -> np.ndarray:
    """Row b = matched prefix slots of request b, then its new slots, padded with -1."""
    b = len(prefix_slots)
    out = np.full((b, stride), -1, np.int32)
    for i in range(b):
        row = np.concatenate([np.asarray(prefix_slots[i], np.int32), np.asarray(new_slots[i], np.int32)])
        out[i, : len(row)] = row
    return out
