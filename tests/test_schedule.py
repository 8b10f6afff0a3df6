"""Cache-aware scheduling and the trace replay (host only) against the oracle's cache model.

"SGLang: Efficient Execution of Structured Language Model Programs": an LRU radix cache under
memory pressure, cache-aware scheduling, hit rates against the optimal one.  The library's
replay (`prefix_cached_kv_radix_gb300.schedule.simulate`) is re-run here decision by decision on
the oracle's dictionary model of the cache: peeked match lengths, evictions, hits, computed
tokens and the final free list must all agree.
"""
import numpy as np
import pytest

import workloads as W
from oracle import PrefixCacheModel
from prefix_cached_kv_radix_gb300 import api, schedule

api.load()


def _oracle_simulate(trace, pool, batch, policy, window=64, seed=0):
    """The replay of `schedule.simulate`, step for step, on the oracle's cache model."""
    m = PrefixCacheModel(pool, seed)
    S = len(trace.sessions)
    nxt, ready_at = [0] * S, [s.start for s in trace.sessions]
    total = sum(len(s.turns) for s in trace.sessions)
    out = dict(requests=0, prompt=0, hit=0, computed=0, evicted=0)
    step = 0
    while out["requests"] < total:
        ready = sorted((ready_at[s], s) for s in range(S) if nxt[s] < len(trace.sessions[s].turns)
                       and ready_at[s] <= step)
        if not ready:
            step = min(ready_at[s] for s in range(S) if nxt[s] < len(trace.sessions[s].turns))
            continue
        cand = [s for _, s in ready]
        reqs = [trace.request(s, nxt[s]) for s in cand]
        if policy == "cache_aware":
            lens = [m._cached_len(list(r)) for r in reqs[:window]]
            order = sorted(range(len(lens)), key=lambda i: (-lens[i], i)) + list(range(len(lens), len(cand)))
        else:
            order = list(range(len(cand)))
        chosen = order[:batch]
        seqs = [list(trace.sequence(cand[i], nxt[cand[i]])) for i in chosen]
        peek = [m._cached_len(q) for q in seqs]
        n_new = [len(q) - k for q, k in zip(seqs, peek)]
        while len(m.alloc.free) < sum(n_new):
            ev = len(m.evict(sum(n_new) - len(m.alloc.free)))
            out["evicted"] += ev
            peek = [m._cached_len(q) for q in seqs]
            n_new = [len(q) - k for q, k in zip(seqs, peek)]
            if ev == 0:
                break
        while sum(n_new) > len(m.alloc.free) and len(chosen) > 1:
            chosen, seqs, peek, n_new = chosen[:-1], seqs[:-1], peek[:-1], n_new[:-1]
        # plan: match (stamps, cuts), allocate, pin; finish: insert, free duplicates, unpin
        matched = []
        for q in seqs:
            k, sl = m.match(q)
            matched.append((k, sl))
        new = m.alloc.alloc(sum(n_new))
        for q, (k, _) in zip(seqs, matched):
            m.lock(q, k)
        off = 0
        dups = []
        for q, (k, sl), nn in zip(seqs, matched, n_new):
            full = np.concatenate([sl, new[off:off + nn]]).astype(np.int32)
            dups.append(m.insert(q, full))
            off += nn
        off = 0
        for q, (k, _), nn, d in zip(seqs, matched, n_new, dups):
            if d > k:
                m.alloc.release(new[off:off + (d - k)])
            off += nn
        for q, (k, _) in zip(seqs, matched):
            m.lock(q, k, -1)
        for j, i in enumerate(chosen):
            s = cand[i]
            rlen = len(reqs[i])
            out["prompt"] += rlen
            out["hit"] += min(peek[j], rlen)
            out["computed"] += n_new[j]
            nxt[s] += 1
            ready_at[s] = step + 1
            out["requests"] += 1
        step += 1
    return out, m


@pytest.mark.parametrize("policy", ["fifo", "cache_aware"])
@pytest.mark.parametrize("pool_frac", [0.2, 0.5])
def test_replay_matches_oracle_model(policy, pool_frac):
    tr = W.chat_trace(3, vocab=64, n_system=2, n_fewshot=2, n_chats=10, n_questions=14, horizon=3, scale=32)
    opt = schedule.optimal(tr)
    longest = max(len(tr.sequence(s, t)) for s in range(len(tr.sessions)) for t in range(len(tr.sessions[s].turns)))
    pool = max(int(pool_frac * opt.computed_tokens), 4 * longest)
    r = schedule.simulate(tr, pool, batch=4, policy=policy)
    o, m = _oracle_simulate(tr, pool, 4, policy)
    assert (r.requests, r.prompt_tokens, r.hit_tokens, r.computed_tokens, r.evicted_tokens) == \
        (o["requests"], o["prompt"], o["hit"], o["computed"], o["evicted"])
    assert r.evicted_tokens > 0                      # the pool was under pressure
    assert r.hit_tokens <= opt.hit_tokens


def test_match_prefix_len_is_read_only():
    rng = np.random.default_rng(5)
    t1, t2 = api.RadixTree(512, 9), api.RadixTree(512, 9)
    m = PrefixCacheModel(512, 9)
    for _ in range(40):
        q = rng.integers(0, 3, size=int(rng.integers(1, 12))).astype(np.int32)
        assert t1.match_prefix_len(q) == m._cached_len(list(q))
        before = t1.stats()
        t1.match_prefix_len(q)
        assert t1.stats() == before                   # no split, no statistics
        if rng.random() < 0.6 and t1.stats()["free_slots"] >= len(q):
            for t in (t1, t2):
                sl = t.alloc_slots(len(q))
                d, _ = t.insert(q, sl)
                t.free_slots(sl[:d])
            sl = m.alloc.alloc(len(q))
            d = m.insert(list(q), sl)
            m.alloc.release(sl[:d])
    # t2 saw the same inserts without the peeks: identical eviction order (no stamps either)
    assert t1.evict(10 ** 6).tolist() == t2.evict(10 ** 6).tolist()
    t1.check()


def test_cache_aware_order_and_hit_bounds():
    tr = W.chat_trace(1, n_chats=120, n_questions=240, horizon=8, scale=4)
    opt = schedule.optimal(tr)
    assert 0.0 < opt.hit_rate < 1.0
    longest = max(len(tr.sequence(s, t)) for s in range(len(tr.sessions)) for t in range(len(tr.sessions[s].turns)))
    pool = max(int(0.5 * opt.computed_tokens), 8 * longest)
    fifo = schedule.simulate(tr, pool, batch=8, policy="fifo")
    aware = schedule.simulate(tr, pool, batch=8, policy="cache_aware")
    for r in (fifo, aware):
        assert r.hit_tokens <= opt.hit_tokens and r.requests == opt.requests
        assert r.prompt_tokens == opt.prompt_tokens
    assert aware.hit_tokens >= fifo.hit_tokens       # ordering by cached prefix pays under pressure
    # with room for everything the order cannot matter beyond a batch's own duplicates
    big = schedule.simulate(tr, opt.computed_tokens * 2, batch=1, policy="cache_aware")
    assert big.hit_tokens == opt.hit_tokens and big.evicted_tokens == 0
    # the order helper itself: longest cached prefix first, ties by position
    t = api.RadixTree(256, 0)
    sl = t.alloc_slots(6)
    t.insert([1, 2, 3, 4, 5, 6], sl)
    assert schedule.cache_aware_order(t, [np.array([9, 9]), np.array([1, 2, 7]), np.array([1, 2, 3, 4]),
                                          np.array([1, 5])]) == [2, 1, 3, 0]


# ---------------------------------------------------------------- offline reference at the same pool
def _steps(*seqs):
    """One request per step, no reply: (request, sequence) pairs from token lists."""
    return [[(np.array(q, np.int32), np.array(q, np.int32))] for q in seqs]


def test_furthest_next_use_hand_worked():
    # pool 4: s0 [1,2] and s1 [3,4] fill it; s2 [5,6] needs 2 slots.  LRU would evict [1,2]
    # (least recent) and miss it at s3; furthest next use evicts 34 (never used again), then its
    # parent 3 (a leaf now, never used again), and s3 [1,2] hits both tokens.
    steps = _steps([1, 2], [3, 4], [5, 6], [1, 2])
    r = schedule.furthest_next_use_replay(steps, 4)
    assert (r.prompt_tokens, r.hit_tokens, r.computed_tokens, r.evicted_tokens) == (8, 2, 6, 2)
    # the library's LRU tree on the same steps: s2 evicts [1,2], s3 misses
    t = api.RadixTree(4, 0)
    hits = 0
    for ((q, _),) in steps:
        slots, m, _ = t.match_prefix(q)
        hits += m
        free = t.stats()["free_slots"]
        if free < len(q) - m:
            t.evict_count(len(q) - m - free)
            slots, m, _ = t.match_prefix(q)
        t.insert(q, np.concatenate([slots[:m], t.alloc_slots(len(q) - m)]).astype(np.int32))
    assert hits == 0


def test_furthest_next_use_token_granular_hand_worked():
    # pool 5.  s0 [1,2,3] computes 3; s1 [1,4] hits 1 (token 1), computes 1 -> cache {1,12,123,14}.
    # s2 [7,8] needs 2, 1 free -> evict 1: the leaves are 123 (depth 3) and 14 (depth 2); the
    # future is s3 [1,2,9] (uses 1 and 12 only), so both leaves are never used again and the
    # deeper one goes: 123.  s3 [1,2,9] hits 2, needs 1, 0 free -> evict 1 among the leaves 14
    # (never again), 78 (never again), 12 (now): equal next use for 14 and 78, equal depth, the
    # later-created one (78) goes.  s4 [1,4] hits 2.
    steps = _steps([1, 2, 3], [1, 4], [7, 8], [1, 2, 9], [1, 4])
    r = schedule.furthest_next_use_replay(steps, 5)
    assert r.prompt_tokens == 3 + 2 + 2 + 3 + 2
    assert r.hit_tokens == 0 + 1 + 0 + 2 + 2
    assert r.computed_tokens == 3 + 1 + 2 + 1 + 0
    assert r.evicted_tokens == 2


def test_offline_reference_bounds():
    tr = W.chat_trace(1, n_chats=60, n_questions=120, horizon=8, scale=4)
    opt = schedule.optimal(tr)
    longest = max(len(tr.sequence(s, t)) for s in range(len(tr.sessions)) for t in range(len(tr.sessions[s].turns)))
    # with room for everything: no eviction, and the same hits as the arrival-order replay in the
    # library (the batches are the same, within-batch duplicates count alike)
    big = opt.computed_tokens * 2
    off = schedule.offline_optimal(tr, big, batch=8)
    lru = schedule.simulate(tr, big, batch=8, policy="fifo")
    assert off.evicted_tokens == 0 and lru.evicted_tokens == 0
    assert (off.requests, off.prompt_tokens, off.hit_tokens, off.computed_tokens) == \
        (lru.requests, lru.prompt_tokens, lru.hit_tokens, lru.computed_tokens)
    # under pressure: never above the unbounded cache, and the batches are the arrival order's
    pool = max(int(0.3 * opt.computed_tokens), 8 * longest)
    off = schedule.offline_optimal(tr, pool, batch=8)
    assert off.evicted_tokens > 0 and off.hit_tokens <= opt.hit_tokens
    assert off.requests == opt.requests and off.prompt_tokens == opt.prompt_tokens
    assert sum(len(b) for b in schedule.fifo_batches(tr, 8)) == opt.requests
