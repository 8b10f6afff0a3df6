"""Native step runtime (rx_step_plan / rx_step_finish) against the oracle's prefix-cache model.

Host code only: a step's match, allocation, pinning, index layout, shared-prefix groups,
insert, free of duplicate slots, eviction and unpinning must equal the same operations
replayed on the oracle, bit for bit, over multi-step scripts.  The host-buffer pipeline's
request ranges (rx_step_ranges, the cuts rx_step_prefetch and rx_step_launch make) are checked
against the policy the header states, restated here.
"""
import numpy as np
import pytest

from oracle import PrefixCacheModel, shared_groups
from prefix_cached_kv_radix_gb300 import api

api.load()


def _stage(batch, total):
    n = api.rx_step_stage_bytes(batch, total)
    buf = np.zeros(n + 64, np.uint8)
    addr = buf.ctypes.data
    return buf, addr, n


def _view(buf, off, n, dt):
    return buf[off:off + n * np.dtype(dt).itemsize].view(dt)


def _auto_ok(gof, glen, P, n_new, heads_per_kv, max_kv):
    if len(glen) == 0 or (gof < 0).any():
        return False
    if n_new.max() * heads_per_kv <= 8 and max_kv <= 1024:     # the small-extend shape: no stacking
        return False
    shared = glen[gof]
    return bool((P + n_new - shared).max() <= 256 and (n_new * heads_per_kv).max() < 128)


def _step(t, m, prompts, n_new, mode, hpk, min_shared, evict_tokens):
    b = len(prompts)
    tok_indptr = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
    tokens = np.concatenate(prompts).astype(np.int32) if b else np.zeros(0, np.int32)
    n_new = np.asarray(n_new, np.int32)
    buf, addr, cap = _stage(b, int(tok_indptr[-1]))
    last = np.empty(max(b, 1), np.int64)
    L = api.rx_step_plan(t.h, tokens, tok_indptr, n_new, mode, hpk, min_shared, addr, cap, last)
    # oracle: match every prompt, allocate, lock
    P, pre = [], []
    for p in prompts:
        k, s = m.match(p)
        P.append(k)
        pre.append(s)
    P = np.array(P, np.int64)
    T = int(n_new.sum())
    new = m.alloc.alloc(T)
    for p, k in zip(prompts, P):
        m.lock(p, int(k))
    assert L.batch == b and L.total_new == T and L.total_prefix == int(P.sum())
    assert L.max_qo_len == (int(n_new.max()) if b else 0)
    assert L.max_kv_len == max([len(p) for p in prompts] + [1]) and L.stride % 8 == 0 and L.stride >= L.max_kv_len
    for off in (L.off_prefix_slots, L.off_prefix_indptr, L.off_new_slots, L.off_qo_indptr, L.off_prefix_lens,
                L.off_kv_lens, L.off_grp_indptr, L.off_grp_members, L.off_grp_len):
        assert off % 256 == 0
    assert L.bytes <= cap
    assert _view(buf, L.off_prefix_slots, L.total_prefix, np.int32).tolist() == \
        (np.concatenate(pre).tolist() if b else [])
    assert _view(buf, L.off_prefix_indptr, b + 1, np.int64).tolist() == [0] + np.cumsum(P).tolist()
    assert _view(buf, L.off_new_slots, T, np.int32).tolist() == new.tolist()
    assert _view(buf, L.off_qo_indptr, b + 1, np.int64).tolist() == [0] + np.cumsum(n_new).tolist()
    assert _view(buf, L.off_prefix_lens, b, np.int32).tolist() == P.tolist()
    assert _view(buf, L.off_kv_lens, b, np.int32).tolist() == (P + n_new).tolist()
    # groups
    gof, glen = shared_groups([p[:k] for p, k in zip(prompts, P)], min_shared)
    use = mode != api.RX_GROUPS_NONE and len(glen) > 0
    if mode == api.RX_GROUPS_AUTO:
        use = use and _auto_ok(gof, glen, P, n_new.astype(np.int64), hpk, max([len(p) for p in prompts] + [1]))
    if use:
        assert L.num_groups == len(glen)
        gi = _view(buf, L.off_grp_indptr, L.num_groups + 1, np.int32)
        gm = _view(buf, L.off_grp_members, int(gi[-1]), np.int32)
        gl = _view(buf, L.off_grp_len, L.num_groups, np.int32)
        assert gl.tolist() == glen.tolist()
        for g in range(L.num_groups):
            assert gm[gi[g]:gi[g + 1]].tolist() == np.flatnonzero(gof == g).tolist()
        assert L.max_group_size == int(np.diff(gi).max()) and L.max_group_len == int(glen.max())
        assert L.max_group_rows == max(int(n_new[gof == g].sum()) for g in range(len(glen)))
    else:
        assert L.num_groups == 0
    # pinned: an eviction of everything leaves the matched prefixes
    # finish on both
    evicted = api.rx_step_finish(t.h, tokens, tok_indptr, last, addr, L, evict_tokens)
    qo = np.concatenate([[0], np.cumsum(n_new)])
    dups = []
    for i, p in enumerate(prompts):
        full = np.concatenate([pre[i], new[qo[i]:qo[i + 1]]]).astype(np.int32)
        dups.append(m.insert(p, full))
    for i in range(b):
        over = dups[i] - P[i]
        if over > 0:
            m.alloc.release(new[qo[i]:qo[i] + over])
    freed = m.evict(evict_tokens) if evict_tokens else np.zeros(0, np.int32)
    for p, k in zip(prompts, P):
        m.lock(p, int(k), -1)
    assert evicted == len(freed)
    st = t.stats()
    assert st["cached_tokens"] == m.cached_tokens() and st["free_slots"] == len(m.alloc.free)
    assert st["node_count"] == len(m.nodes())
    t.check()


def _random_prompts(rng, m, b, vocab, maxlen):
    """Prompts whose last n_new tokens are exactly the uncached tail (distinct first new token
    per divergence point, so that no earlier request of the batch caches a later one's tail)."""
    prompts, n_new, used = [], [], set()
    for _ in range(b):
        for _try in range(50):
            p = rng.integers(0, vocab, size=int(rng.integers(1, maxlen + 1))).tolist()
            k = m._cached_len(p)
            if k == len(p) and rng.random() < 0.7:
                continue
            key = (tuple(p[:k]), p[k] if k < len(p) else None)
            if key in used:
                continue
            used.add(key)
            prompts.append(np.array(p, np.int32))
            n_new.append(len(p) - k)
            break
    return prompts, n_new


@pytest.mark.parametrize("mode", [api.RX_GROUPS_NONE, api.RX_GROUPS_ALWAYS, api.RX_GROUPS_AUTO])
def test_step_scripts_match_oracle(mode):
    rng = np.random.default_rng(40 + mode)
    for trial in range(6):
        t = api.RadixTree(600, trial)
        m = PrefixCacheModel(600, trial)
        for step in range(8):
            prompts, n_new = _random_prompts(rng, m, int(rng.integers(0, 7)), 3, 12)
            if sum(n_new) > len(m.alloc.free):
                break
            _step(t, m, prompts, n_new, mode, int(rng.choice([1, 4, 16])), int(rng.integers(1, 4)),
                  int(rng.integers(0, 10)))
        n = t.stats()["free_slots"]
        assert t.alloc_slots(n).tolist() == m.alloc.alloc(n).tolist()


def test_step_plan_rejects_cached_tail_without_side_effects():
    t = api.RadixTree(64, 2)
    s = t.alloc_slots(4)
    t.insert([1, 2, 3, 4], s)
    before = t.stats()
    tokens = np.array([1, 2, 3, 4, 5], np.int32)
    ind = np.array([0, 5], np.int64)
    buf, addr, cap = _stage(1, 5)
    last = np.empty(1, np.int64)
    with pytest.raises(api.RxError) as e:      # claims 2 new tokens; only 1 is uncached
        api.rx_step_plan(t.h, tokens, ind, np.array([2], np.int32), 0, 1, 1, addr, cap, last)
    assert e.value.code == api.RX_EINVAL
    after = t.stats()
    assert after["free_slots"] == before["free_slots"] and after["cached_tokens"] == before["cached_tokens"]
    # nothing was pinned: everything is still evictable
    assert len(t.evict(100)) == 4
    t.check()


def test_step_plan_out_of_slots_and_small_stage():
    t = api.RadixTree(8, 0)
    tokens = np.arange(10, dtype=np.int32)
    ind = np.array([0, 10], np.int64)
    buf, addr, cap = _stage(1, 10)
    last = np.empty(1, np.int64)
    with pytest.raises(api.RxError) as e:
        api.rx_step_plan(t.h, tokens, ind, np.array([10], np.int32), 0, 1, 1, addr, cap, last)
    assert e.value.code == api.RX_ENOMEM
    assert t.stats()["free_slots"] == 8
    with pytest.raises(api.RxError) as e:
        api.rx_step_plan(t.h, tokens[:4], np.array([0, 4], np.int64), np.array([4], np.int32), 0, 1, 1, addr,
                         16, last)
    assert e.value.code == api.RX_EINVAL


def test_step_pins_prefixes_until_finish():
    t = api.RadixTree(64, 5)
    s = t.alloc_slots(6)
    t.insert([7, 7, 7, 7, 7, 7], s)
    tokens = np.array([7, 7, 7, 7, 7, 7, 8, 9], np.int32)
    ind = np.array([0, 8], np.int64)
    buf, addr, cap = _stage(1, 8)
    last = np.empty(1, np.int64)
    L = api.rx_step_plan(t.h, tokens, ind, np.array([2], np.int32), 0, 1, 1, addr, cap, last)
    assert len(t.evict(100)) == 0            # the matched prefix is pinned
    ev = api.rx_step_finish(t.h, tokens, ind, last, addr, L, 100)
    assert ev == 2 and t.stats()["cached_tokens"] == 6   # evicts before unpinning: only the new leaf
    assert len(t.evict(100)) == 6                        # unpinned afterwards
    t.check()


def test_long_prompt_step_equals_per_call_replay():
    """Prompts long enough (here ~130 K tokens a step) for rx_step_plan to read them against the
    tree on its worker threads.  The matched slots must equal the oracle's list matcher, and the
    whole step -- stamps, splits, node ids, allocation, insert, eviction order -- must equal the
    same step replayed through the single-call entry points (match_prefix per request, lock,
    insert_batch_at, evict, unlock) on a twin tree."""
    from oracle import ListMatcher
    rng = np.random.default_rng(77)
    vocab = 50000
    root = rng.integers(0, vocab, size=4000).astype(np.int32)
    branches = [np.concatenate([root, rng.integers(0, vocab, size=3000).astype(np.int32)]) for _ in range(4)]
    t1, t2 = api.RadixTree(1 << 16, 5), api.RadixTree(1 << 16, 5)
    lm = ListMatcher()
    for br in branches:
        for t in (t1, t2):
            k = t.match_prefix_len(br)
            sl = t.alloc_slots(len(br) - k)
            full = np.concatenate([np.zeros(k, np.int32), sl]).astype(np.int32)
            d, _ = t.insert(br, full)
        k, pre = lm.match(br)
        lm.add(br, np.concatenate([pre, sl]).astype(np.int32))
    for step in range(3):
        prompts, n_new = [], []
        for b in range(24):
            br = branches[b % 4]
            cached = t1.match_prefix_len(br)            # eviction trims the branches step by step
            cut = int(rng.integers(1, cached + 1))
            n = int(rng.integers(1, 4))
            tail = rng.integers(vocab, vocab + 10 ** 6, size=n).astype(np.int32)   # never cached
            prompts.append(np.concatenate([br[:cut], tail]))
            n_new.append(n)
        tok_indptr = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
        tokens = np.concatenate(prompts).astype(np.int32)
        assert tok_indptr[-1] > (1 << 15)
        nn = np.asarray(n_new, np.int32)
        T = int(nn.sum())
        buf, addr, cap = _stage(len(prompts), int(tok_indptr[-1]))
        last = np.empty(len(prompts), np.int64)
        L = api.rx_step_plan(t1.h, tokens, tok_indptr, nn, api.RX_GROUPS_NONE, 1, 1, addr, cap, last)
        got = _view(buf, L.off_prefix_slots, L.total_prefix, np.int32)
        P = _view(buf, L.off_prefix_lens, len(prompts), np.int32).copy()
        want = [lm.match(p) for p in prompts]
        assert P.tolist() == [k for k, _ in want]
        assert got.tolist() == np.concatenate([s for _, s in want]).tolist()
        evicted1 = api.rx_step_finish(t1.h, tokens, tok_indptr, last, addr, L, T)
        # the same step through the single-call entry points
        lasts, slots2 = [], []
        for p in prompts:
            s2, k2, n2 = t2.match_prefix(p)
            lasts.append(n2)
            slots2.append(s2)
        assert lasts == last.tolist()
        assert np.concatenate(slots2).tolist() == got.tolist()
        new = t2.alloc_slots(T)
        assert new.tolist() == _view(buf, L.off_new_slots, T, np.int32).tolist()
        api.radix_lock_batch(t2.h, lasts)
        qo = np.concatenate([[0], np.cumsum(nn)]).astype(np.int64)
        dups, _ = api.insert_batch_at(t2.h, lasts, tokens, tok_indptr, new, qo)
        for b, d in enumerate(dups):
            if d > P[b]:
                t2.free_slots(new[qo[b]:qo[b] + d - P[b]])
        freed2 = t2.evict(T)
        api.radix_unlock_batch(t2.h, lasts)
        assert evicted1 == len(freed2)
        assert t1.stats() == t2.stats()
        for p in prompts:
            lm.add(p, np.concatenate([lm.match(p)[1], np.zeros(len(p) - lm.match(p)[0], np.int32)]))
        t1.check()
    # identical stamps and structure: everything evicts in the same order
    assert t1.evict(10 ** 7).tolist() == t2.evict(10 ** 7).tolist()


# ---------------------------------------------------------------- host-buffer pipeline ranges
def _expected_ranges(n_new, hq, hkv, d, elt, chunks):
    """The pipeline's cuts restated from the header: `chunks` ranges of about equal token counts
    (range c starts at the first request whose rows start at or after c/n of the tokens), or,
    for chunks = 0, one range per 64 MB of rows moved (at most 4) with the last eighth of the
    last range's tokens (at least one request) split off when there are several."""
    B = len(n_new)
    qo = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int64)
    T = int(qo[-1])
    moved = T * (2 * hq * d * elt + 2 * hkv * d * elt)
    nc = chunks if chunks > 0 else min(4, max(1, moved >> 26))
    nc = max(1, min(nc, max(B, 1)))
    cut = [0]
    for c in range(1, nc):
        target = T * c // nc
        first = next((b for b in range(B) if qo[b] >= target), B)
        cut.append(max(first, cut[-1]))
    cut.append(B)
    if chunks <= 0 and nc > 1 and B - cut[-2] >= 2:
        b0 = cut[-2]
        target = qo[B] - (qo[B] - qo[b0]) // 8
        s = next((b for b in range(b0 + 1, B) if qo[b] >= target), B)
        cut.insert(len(cut) - 1, min(s, B - 1))
    return np.asarray(cut, np.int32)


@pytest.mark.parametrize("shape", [(64, 8, 128, 2), (32, 8, 128, 2), (12, 12, 64, 2), (4, 4, 64, 4)])
@pytest.mark.parametrize("chunks", [0, 1, 3, 4, 8])
def test_step_ranges_follow_the_stated_policy(shape, chunks):
    hq, hkv, d, elt = shape
    desc = api.make_desc(api.RX_F32 if elt == 4 else api.RX_BF16, hq, hkv, d, 1 << 22, d ** -0.5)
    rng = np.random.default_rng(hq * 100 + chunks)
    cases = [[1024] * 32, [128] * 128, [800] * 9 + [0], [0, 0, 5000, 0, 3000, 0], [7, 8] * 32, [], [3],
             list(rng.integers(0, 3000, size=57)), [20000, 1, 1, 1], [1, 1, 1, 20000]]
    for n_new in cases:
        got = api.rx_step_ranges(desc, np.asarray(n_new, np.int32), chunks)
        want = _expected_ranges(np.asarray(n_new, np.int64), hq, hkv, d, elt, chunks)
        assert np.array_equal(got, want), (n_new[:8], got, want)
        assert got[0] == 0 and got[-1] == len(n_new) and (np.diff(got) >= 0).all()


def test_step_ranges_at_the_benchmark_shapes():
    """c5 (32 x 1024 new rows, 64/8 heads x 128): four ranges of 8 requests with the last one's
    final request on its own; c3 (128 x 128, 32/8 x 128): the last 4 requests on their own."""
    c5 = api.make_desc(api.RX_BF16, 64, 8, 128, 1 << 22, 128 ** -0.5)
    assert api.rx_step_ranges(c5, [1024] * 32).tolist() == [0, 8, 16, 24, 31, 32]
    assert api.rx_step_ranges(c5, [1024] * 32, 4).tolist() == [0, 8, 16, 24, 32]
    c3 = api.make_desc(api.RX_BF16, 32, 8, 128, 1 << 20, 128 ** -0.5)
    assert api.rx_step_ranges(c3, [128] * 128).tolist() == [0, 32, 64, 96, 124, 128]
    c2 = api.make_desc(api.RX_BF16, 12, 12, 64, 1 << 16, 64 ** -0.5)
    assert api.rx_step_ranges(c2, [8] * 64).tolist() == [0, 64]          # 3 MB: one range


def test_step_ranges_reject_bad_arguments():
    desc = api.make_desc(api.RX_BF16, 32, 8, 128, 1 << 20, 128 ** -0.5)
    with pytest.raises(RuntimeError):
        api.rx_step_ranges(desc, np.asarray([5, -1, 3], np.int32))
    lib = api.load()
    nn = np.asarray([128] * 128, np.int32)
    cuts = np.zeros(3, np.int32)
    n = np.zeros(1, np.int32)
    assert lib.rx_step_ranges(api.ctypes.byref(desc), len(nn), nn.ctypes.data, 0, cuts.ctypes.data, 3,
                              n.ctypes.data) == api.RX_EINVAL
