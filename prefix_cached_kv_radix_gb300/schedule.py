"""Cache-aware scheduling, and a replay of request traces through the radix cache (host only).

"SGLang: Efficient Execution of Structured Language Model Programs": RadixAttention keeps an
LRU cache of KV in a radix tree and evicts least-recently-used nodes under memory pressure (the
nine-step walk-through); the runtime's scheduling is cache-aware, and the results report cache
hit rates of 50-99% and 96% of the optimal hit rate.

`simulate` replays a trace (`workloads.Trace`) through the library's tree and allocator under a
pool of bounded size: each step takes a batch of waiting requests (in arrival order, or
cache-aware: longest cached prefix first within a window of waiting requests), evicts LRU leaves
when the batch's new tokens do not fit, plans the step (match, allocate, pin) and finishes it
(insert the request and its reply, unpin), exactly as a serving step does, but allocates slots
only: no K/V is computed.  Two references: the hit rate of an unbounded cache (every distinct
prefix token computed once, whatever the order: no policy reaches it under a bounded pool), and
an offline replay of the arrival order at the same pool size that evicts by furthest next use
(Belady's rule, knowing the future requests: `offline_optimal`).

    python -m prefix_cached_kv_radix_gb300.schedule [--seed 1] [--batch 8] [--chats 400] [--questions 800]

prints the hit rates of both orders at several pool sizes against both references.
"""
from __future__ import annotations

import argparse
from dataclasses import dataclass

import numpy as np

from . import api


def cache_aware_order(tree: api.RadixTree, prompts) -> list:
    """Indices of `prompts` by decreasing cached-prefix length, ties in the given order (a
    read-only query of the tree: no LRU stamp, no split)."""
    if not len(prompts):
        return []
    ind = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
    lens = tree.match_prefix_len_batch(np.concatenate(prompts).astype(np.int32), ind)
    return sorted(range(len(prompts)), key=lambda i: (-int(lens[i]), i))


@dataclass
class TraceResult:
    requests: int = 0
    prompt_tokens: int = 0           # tokens of the requests (replies excluded)
    hit_tokens: int = 0              # request tokens found in the cache
    computed_tokens: int = 0         # tokens that had to be computed (uncached request tokens + replies)
    evicted_tokens: int = 0
    steps: int = 0

    @property
    def hit_rate(self) -> float:
        return self.hit_tokens / max(self.prompt_tokens, 1)


def simulate(trace, pool_slots: int, batch: int = 8, policy: str = "fifo", window: int = 64,
             seed: int = 0, page_size: int = 1) -> TraceResult:
    """Replay every turn of every session of `trace`; a session's next turn becomes ready the
    step after its previous turn (its prompt holds that turn's reply).  With page_size > 1
    only whole pages of a match are reused."""
    assert policy in ("fifo", "cache_aware")
    tree = api.RadixTree(pool_slots, seed, page_size=page_size)
    S = len(trace.sessions)
    nxt = [0] * S
    ready_at = [s.start for s in trace.sessions]
    total = sum(len(s.turns) for s in trace.sessions)
    res = TraceResult()
    step = 0
    stage = np.zeros(0, np.uint8)
    while res.requests < total:
        ready = sorted((ready_at[s], s) for s in range(S) if nxt[s] < len(trace.sessions[s].turns)
                       and ready_at[s] <= step)
        if not ready:
            step = min(ready_at[s] for s in range(S) if nxt[s] < len(trace.sessions[s].turns))
            continue
        cand = [s for _, s in ready]
        reqs = [trace.request(s, nxt[s]) for s in cand]
        if policy == "cache_aware":
            order = cache_aware_order(tree, reqs[:window])
            order += list(range(len(order), len(cand)))
        else:
            order = list(range(len(cand)))
        chosen = order[:batch]
        seqs = [trace.sequence(cand[i], nxt[cand[i]]) for i in chosen]
        ind = np.concatenate([[0], np.cumsum([len(q) for q in seqs])]).astype(np.int64)
        toks = np.concatenate(seqs).astype(np.int32)
        m = tree.match_prefix_len_batch(toks, ind)
        n_new = np.array([len(q) for q in seqs], np.int64) - m
        free = tree.stats()["free_slots"]
        while free < n_new.sum():        # memory pressure: free LRU leaves (none is pinned now)
            ev = tree.evict_count(int(n_new.sum()) - free)
            res.evicted_tokens += ev
            m = tree.match_prefix_len_batch(toks, ind)   # eviction may have taken part of a match
            n_new = np.array([len(q) for q in seqs], np.int64) - m
            free = tree.stats()["free_slots"]
            if ev == 0:
                break
        while n_new.sum() > free and len(chosen) > 1:      # still too big: run fewer requests
            chosen, seqs = chosen[:-1], seqs[:-1]
            ind = ind[:len(seqs) + 1]
            toks = toks[:ind[-1]]
            m, n_new = m[:len(seqs)], n_new[:len(seqs)]
        need = api.rx_step_stage_bytes(len(seqs), int(ind[-1]))
        if stage.nbytes < need:
            stage = np.zeros(2 * need, np.uint8)
        last = np.empty(len(seqs), np.int64)
        lay = api.rx_step_plan(tree.h, toks, ind, n_new.astype(np.int32), api.RX_GROUPS_NONE, 1, 1,
                               stage.ctypes.data, stage.nbytes, last)
        api.rx_step_finish(tree.h, toks, ind, last, stage.ctypes.data, lay, 0)
        for k, i in enumerate(chosen):
            s = cand[i]
            rlen = len(reqs[i])
            res.prompt_tokens += rlen
            res.hit_tokens += int(min(m[k], rlen))
            res.computed_tokens += int(n_new[k])
            nxt[s] += 1
            ready_at[s] = step + 1
            res.requests += 1
        res.steps += 1
        step += 1
    tree.check()
    return res


def fifo_batches(trace, batch: int) -> list:
    """The batches of (session, turn) that simulate(policy="fifo") runs when no batch has to
    shrink for lack of room (the arrival order does not depend on the cache's contents)."""
    S = len(trace.sessions)
    nxt = [0] * S
    ready_at = [s.start for s in trace.sessions]
    total = sum(len(s.turns) for s in trace.sessions)
    out, done, step = [], 0, 0
    while done < total:
        ready = sorted((ready_at[s], s) for s in range(S) if nxt[s] < len(trace.sessions[s].turns)
                       and ready_at[s] <= step)
        if not ready:
            step = min(ready_at[s] for s in range(S) if nxt[s] < len(trace.sessions[s].turns))
            continue
        chosen = [s for _, s in ready][:batch]
        out.append([(s, nxt[s]) for s in chosen])
        for s in chosen:
            nxt[s] += 1
            ready_at[s] = step + 1
            done += 1
        step += 1
    return out


def furthest_next_use_replay(steps, pool_slots: int) -> TraceResult:
    """Offline replay of a fixed sequence of steps under a pool of `pool_slots` token slots,
    evicting by furthest next use (Belady's rule for paging, applied to cached tokens).

    steps: list of steps, each a list of (request_tokens, sequence_tokens) where the sequence is
    the request followed by its reply (what the cache holds after the step).  Each cached token
    is one prefix (a node of the trie of all sequences).  Per step, as in `simulate`: every
    sequence's cached prefix is looked up before the step, hits = cached tokens of the request
    part, the uncached tokens are computed; when they do not fit in the free slots, cached
    tokens are evicted one at a time from the ends of cached paths (a token with no cached
    extension), the one whose next use (the first step at or after this one whose sequence
    contains it) is furthest first -- never used again counts as infinitely far; ties go to the
    deeper token, then to the later-created one.  Then every sequence is inserted (tokens two
    sequences of a step share are computed by both and stored once)."""
    import bisect
    import heapq
    ids_of = []               # per step, per sequence: the prefix ids of its tokens
    node = {}                 # (parent id, token) -> prefix id
    parent, depth = [], []
    uses = []                 # prefix id -> steps whose sequences contain it (ascending)
    for t, st in enumerate(steps):
        per = []
        for _, seq in st:
            ids = np.empty(len(seq), np.int64)
            p = -1
            for i, tok in enumerate(seq.tolist() if hasattr(seq, "tolist") else seq):
                key = (p, tok)
                q = node.get(key)
                if q is None:
                    q = node[key] = len(parent)
                    parent.append(p)
                    depth.append(i + 1)
                    uses.append([])
                if not uses[q] or uses[q][-1] != t:
                    uses[q].append(t)
                ids[i] = q
                p = q
            per.append(ids)
        ids_of.append(per)
    n = len(parent)
    cached = np.zeros(n, bool)
    nchild = np.zeros(n, np.int64)
    leaves = set()
    free = pool_slots
    res = TraceResult()
    INF = len(steps) + 1

    def cached_len(ids):
        k = 0
        while k < len(ids) and cached[ids[k]]:
            k += 1
        return k

    def key(q, t):
        u = uses[q]
        i = bisect.bisect_left(u, t)
        nu = u[i] if i < len(u) else INF
        return (-nu, -depth[q], -q, q)

    for t, st in enumerate(steps):
        m = [cached_len(ids) for ids in ids_of[t]]
        need = sum(len(ids) - k for ids, k in zip(ids_of[t], m))
        if free < need:
            heap = [key(q, t) for q in leaves]
            heapq.heapify(heap)
            while free < need and heap:
                q = heapq.heappop(heap)[3]
                cached[q] = False
                leaves.discard(q)
                free += 1
                res.evicted_tokens += 1
                p = parent[q]
                if p >= 0:
                    nchild[p] -= 1
                    if nchild[p] == 0:
                        leaves.add(p)
                        heapq.heappush(heap, key(p, t))
            m = [cached_len(ids) for ids in ids_of[t]]
            need = sum(len(ids) - k for ids, k in zip(ids_of[t], m))
        newly = 0
        for ids, k in zip(ids_of[t], m):
            for q in ids[k:].tolist():
                if not cached[q]:
                    cached[q] = True
                    newly += 1
                    leaves.add(q)
                    p = parent[q]
                    if p >= 0:
                        if nchild[p] == 0:
                            leaves.discard(p)
                        nchild[p] += 1
        free -= newly
        assert free >= 0, "pool smaller than one step's new tokens"
        for (req, _), k in zip(st, m):
            res.prompt_tokens += len(req)
            res.hit_tokens += min(k, len(req))
            res.requests += 1
        res.computed_tokens += need
        res.steps += 1
    return res


def offline_optimal(trace, pool_slots: int, batch: int = 8) -> TraceResult:
    """The arrival-order schedule replayed offline at the same pool size with furthest-next-use
    eviction: the reference that the LRU replays' hit rates are compared with at that size."""
    steps = [[(trace.request(s, t), trace.sequence(s, t)) for s, t in b] for b in fifo_batches(trace, batch)]
    return furthest_next_use_replay(steps, pool_slots)


def optimal(trace) -> TraceResult:
    """Hit counts of an unbounded cache (one request at a time): the most any order can reuse."""
    tot = sum(len(trace.sequence(s, t)) for s in range(len(trace.sessions))
              for t in range(len(trace.sessions[s].turns)))
    return simulate(trace, tot + 1, batch=1, policy="fifo")


def main():
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import workloads as W
    ap = argparse.ArgumentParser()
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--window", type=int, default=64)
    ap.add_argument("--chats", type=int, default=400)
    ap.add_argument("--questions", type=int, default=800)
    ap.add_argument("--horizon", type=int, default=16, help="arrivals spread over this many steps")
    a = ap.parse_args()
    tr = W.chat_trace(a.seed, n_chats=a.chats, n_questions=a.questions, horizon=a.horizon)
    opt = optimal(tr)
    distinct = opt.computed_tokens          # every distinct token computed once
    longest = max(len(tr.sequence(s, t)) for s in range(len(tr.sessions)) for t in range(len(tr.sessions[s].turns)))
    print(f"trace: {len(tr.sessions)} sessions, {opt.requests} requests, {opt.prompt_tokens} prompt tokens, "
          f"{distinct} distinct tokens; optimal hit rate {opt.hit_rate:.4f}")
    print()
    print("| pool (share of distinct tokens) | order / eviction | hit rate | % of unbounded | "
          "% of offline at this pool | evicted tokens |")
    print("|---|---|---|---|---|---|")
    for frac in (0.05, 0.1, 0.25, 0.5, 1.0):
        pool = max(int(frac * distinct), a.batch * longest)
        off = offline_optimal(tr, pool, batch=a.batch)
        print(f"| {frac:.2f} ({pool} slots) | arrival / offline furthest next use | {off.hit_rate:.4f} | "
              f"{100 * off.hit_rate / opt.hit_rate:.1f} % | 100 % | {off.evicted_tokens} |")
        for pol in ("fifo", "cache_aware"):
            r = simulate(tr, pool, batch=a.batch, policy=pol, window=a.window)
            print(f"| {frac:.2f} ({pool} slots) | {'arrival' if pol == 'fifo' else 'cache-aware'} / LRU | "
                  f"{r.hit_rate:.4f} | {100 * r.hit_rate / opt.hit_rate:.1f} % | "
                  f"{100 * r.hit_rate / off.hit_rate:.1f} % | {r.evicted_tokens} |")
    # reuse granularity: hits lost at page boundaries (cache-aware order)
    print()
    print("| page size | pool (share of distinct tokens) | hit rate | % of the token-granular optimum | computed tokens |")
    print("|---|---|---|---|---|")
    for frac in (0.5, 1.0):
        pool = max(int(frac * distinct), a.batch * longest)
        for page in (1, 4, 16, 64):
            r = simulate(tr, pool, batch=a.batch, policy="cache_aware", window=a.window, page_size=page)
            print(f"| {page} | {frac:.2f} | {r.hit_rate:.4f} | {100 * r.hit_rate / opt.hit_rate:.1f} % | "
                  f"{r.computed_tokens} |")


if __name__ == "__main__":
    main()
