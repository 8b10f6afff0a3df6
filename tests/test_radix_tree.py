"""Host C++ radix tree (through the C ABI) against the oracle's prefix-cache model.

No GPU needed: the tree and allocator are host code.  Slots, match lengths, dup lengths,
eviction order, node counts and free-list order must be bit-exact against the oracle.
"""
import itertools

import numpy as np
import pytest

from oracle import PrefixCacheModel, slot_order
from prefix_cached_kv_radix_gb300 import api

api.load()


def test_allocator_order_matches_oracle():
    t = api.RadixTree(1000, 123)
    got = t.alloc_slots(1000)
    assert got.tolist() == slot_order(1000, 123).tolist()
    with pytest.raises(api.RxError) as e:
        t.alloc_slots(1)
    assert e.value.code == api.RX_ENOMEM
    t.free_slots(got[[5, 3]])
    assert t.alloc_slots(2).tolist() == [got[5], got[3]]


def test_free_slot_errors_leave_state_unchanged():
    t = api.RadixTree(16, 1)
    s = t.alloc_slots(4)
    with pytest.raises(api.RxError):
        t.free_slots([s[0], s[0]])
    with pytest.raises(api.RxError):
        t.free_slots([s[1], 99])
    assert t.stats()["free_slots"] == 12
    t.free_slots(s)
    assert t.stats()["free_slots"] == 16
    t.check()


def test_insert_rejects_unallocated_slots():
    t = api.RadixTree(16, 1)
    free_slot = int(slot_order(16, 1)[0])
    with pytest.raises(api.RxError):
        t.insert([1, 2], [free_slot, free_slot])
    with pytest.raises(api.RxError):
        t.insert([1], [16])


def test_lock_semantics():
    t = api.RadixTree(64, 0)
    a = t.alloc_slots(3)
    _, na = t.insert([1, 1, 1], a)
    b = t.alloc_slots(3)
    _, nb = t.insert([2, 2, 2], b)
    t.lock(na)
    assert t.evict(100).tolist() == b.tolist()
    assert t.evict(100).tolist() == []
    t.unlock(na)
    with pytest.raises(api.RxError) as e:
        t.unlock(na)
    assert e.value.code == api.RX_ELOCKED
    assert t.evict(1).tolist() == a.tolist()
    with pytest.raises(api.RxError):
        t.lock(na)                     # evicted node: unknown handle
    t.check()


def test_long_edge_matches_up_to_every_divergence_point():
    """Reading a prompt along a long cached edge (compared in blocks of 64 and 16 tokens, then
    token by token) stops exactly at the first differing token, wherever it falls relative to
    the blocks; the read-only and the splitting match agree."""
    edge = np.arange(1, 1001, dtype=np.int32)
    for cut in [0, 1, 2, 15, 16, 17, 63, 64, 65, 79, 80, 127, 128, 129, 500, 998, 999, 1000]:
        t = api.RadixTree(4096, 5)
        sl = t.alloc_slots(len(edge))
        t.insert(edge, sl)
        prompt = np.concatenate([edge[:cut], [-7], edge[cut + 1:]]).astype(np.int32) if cut < 1000 \
            else np.concatenate([edge, [5, 6, 7]]).astype(np.int32)
        assert t.match_prefix_len(prompt) == cut
        got, n, _ = t.match_prefix(prompt)
        assert n == cut and got.tolist() == sl[:cut].tolist()
        t.check()


def test_recycled_nodes_get_new_handles():
    """Evicted nodes are recycled for later inserts (their storage, not their handles): the
    handle of an evicted node stays unknown after its memory holds a new node, new handles
    never repeat, and the tree checks out over many insert/evict rounds."""
    t = api.RadixTree(512, 3)
    rng = np.random.default_rng(7)
    dead, seen = [], set()
    for rnd in range(30):
        live = []
        for i in range(8):                       # eight fresh leaves under distinct first tokens
            toks = [1000 * rnd + i] + rng.integers(0, 9, size=int(rng.integers(1, 6))).tolist()
            sl = t.alloc_slots(len(toks))
            dup, node = t.insert(toks, sl)
            assert dup == 0 and node not in seen
            seen.add(node)
            live.append(node)
        t.check()
        for node in dead[-16:]:                  # handles of nodes whose storage may now be reused
            with pytest.raises(api.RxError):
                t.lock(node)
        assert len(t.evict(10 ** 6)) > 0         # everything goes: the next round reuses it
        dead.extend(live)
        t.check()
    assert t.stats()["node_count"] == 0


def _run_script(ops, num_slots, seed):
    """Apply the same operations to the C++ tree and the oracle model; compare everything."""
    t = api.RadixTree(num_slots, seed)
    m = PrefixCacheModel(num_slots, seed)
    for op, arg in ops:
        if op == "match":
            s1, n1, _ = t.match_prefix(arg)
            n2, s2 = m.match(arg)
            assert n1 == n2 and s1.tolist() == s2.tolist()
        elif op == "insert":
            n_free = t.stats()["free_slots"]
            if n_free < len(arg):
                continue
            new = t.alloc_slots(len(arg))
            new2 = m.alloc.alloc(len(arg))
            assert new.tolist() == new2.tolist()
            d1, _ = t.insert(arg, new)
            d2 = m.insert(arg, new2)
            assert d1 == d2
            t.free_slots(new[:d1])
            m.alloc.release(new2[:d2])
        elif op == "evict":
            f1 = t.evict(arg)
            f2 = m.evict(arg)
            assert f1.tolist() == f2.tolist()
        st = t.stats()
        assert st["node_count"] == len(m.nodes())
        assert st["cached_tokens"] == m.cached_tokens()
        assert st["free_slots"] == len(m.alloc.free)
        t.check()
    # the free lists agree in order too
    n = t.stats()["free_slots"]
    assert t.alloc_slots(n).tolist() == m.alloc.alloc(n).tolist()


@pytest.mark.parametrize("vocab", [2, 3, 4])
def test_random_scripts_match_oracle(vocab):
    rng = np.random.default_rng(100 + vocab)
    for trial in range(25):
        ops = []
        for _ in range(25):
            r = rng.random()
            seq = rng.integers(0, vocab, size=rng.integers(1, 11)).tolist()
            if r < 0.4:
                ops.append(("match", seq))
            elif r < 0.85:
                ops.append(("insert", seq))
            else:
                ops.append(("evict", int(rng.integers(1, 8))))
        _run_script(ops, 48, trial)


def test_wide_fanout_scripts_match_oracle():
    """Hundreds of children under one node (the child links' open-addressing table grows, and
    evictions delete from it with backward shifts, among long probe runs): the tree still
    equals the oracle model op for op."""
    rng = np.random.default_rng(77)
    for trial in range(3):
        ops = []
        for _ in range(400):
            r = rng.random()
            seq = [int(rng.integers(0, 500))] + rng.integers(0, 3, size=rng.integers(0, 5)).tolist()
            if r < 0.3:
                ops.append(("match", seq))
            elif r < 0.85:
                ops.append(("insert", seq))
            else:
                ops.append(("evict", int(rng.integers(1, 40))))
        _run_script(ops, 2000, 50 + trial)


def test_exhaustive_short_sequences():
    seqs = [list(s) for L in range(1, 4) for s in itertools.product([0, 1], repeat=L)]
    ops = []
    for s in seqs:
        ops.append(("insert", s))
    for s in seqs:
        ops.append(("match", s + [2]))
    ops += [("evict", 3), ("match", [0, 1]), ("evict", 5), ("insert", [1, 1, 1, 1]), ("evict", 100)]
    _run_script(ops, 64, 9)


def test_batch_entry_points_equal_single_calls():
    rng = np.random.default_rng(7)
    seqs = [rng.integers(0, 3, size=rng.integers(1, 9)).astype(np.int32) for _ in range(20)]
    t1, t2 = api.RadixTree(512, 3), api.RadixTree(512, 3)
    ind = np.concatenate([[0], np.cumsum([len(s) for s in seqs])])
    flat = np.concatenate(seqs)
    slots = t1.alloc_slots(len(flat))
    assert slots.tolist() == t2.alloc_slots(len(flat)).tolist()
    dups, lasts = t1.insert_batch(flat, ind, slots)
    for i, s in enumerate(seqs):
        d, l = t2.insert(s, slots[ind[i]:ind[i + 1]])
        assert d == dups[i] and l == lasts[i]
    q = [np.concatenate([s, [5]]).astype(np.int32) for s in seqs]
    qind = np.concatenate([[0], np.cumsum([len(s) for s in q])])
    ms, mind, ml = t1.match_prefix_batch(np.concatenate(q), qind)
    for i, s in enumerate(q):
        s2, n2, l2 = t2.match_prefix(s)
        assert mind[i + 1] - mind[i] == n2 and ms[mind[i]:mind[i + 1]].tolist() == s2.tolist() and ml[i] == l2
    assert t1.stats() == t2.stats()


def test_shared_groups():
    t = api.RadixTree(4096, 0)
    shared = list(range(100, 140))                       # 40-token shared prefix
    seqs = [shared + [1000 + i, 7, 7] for i in range(5)] + [[9, 9, 9, 9]] + [shared[:10] + [55]]
    lasts = []
    for s in seqs:
        sl = t.alloc_slots(len(s))
        d, l = t.insert(s, sl)
        t.free_slots(sl[:d])
        lasts.append(l)
    gof, glen = t.shared_groups(lasts, min_shared=1)
    # the five requests share 40 tokens; the 7th shares only 10 with them -> all 6 under
    # one top node with common depth 10; [9,9,9,9] is alone
    assert gof.tolist() == [0, 0, 0, 0, 0, -1, 0] and glen.tolist() == [10]
    gof, glen = t.shared_groups(lasts[:5], min_shared=1)
    assert gof.tolist() == [0] * 5 and glen.tolist() == [40]
    gof, glen = t.shared_groups(lasts[:5], min_shared=41)
    assert gof.tolist() == [-1] * 5 and len(glen) == 0


def test_nine_step_walkthrough_on_the_tree():
    """The walk-through's event script run on the C++ tree and the oracle side by side."""
    SYS = [1, 2, 3, 4]
    ops = [("insert", SYS + [10, 11, 12, 12]),
           ("match", SYS + [10, 11, 12, 12, 13]), ("insert", SYS + [10, 11, 12, 12, 13, 14, 14]),
           ("match", SYS + [20, 21]), ("insert", SYS + [20, 21, 22, 22]),
           ("match", SYS + [20, 21, 22, 22, 23]), ("evict", 3), ("insert", SYS + [20, 21, 22, 22, 23, 24, 24]),
           ("insert", [30, 31, 32, 33, 34, 35, 36]),
           ("insert", [30, 31, 32, 33, 34, 40, 36]), ("insert", [30, 31, 32, 33, 34, 41, 36]),
           ("match", SYS + [10, 11, 12, 12, 15]), ("evict", 4), ("insert", SYS + [10, 11, 12, 12, 15, 16, 16, 16]),
           ("evict", 3), ("insert", SYS + [10, 11, 12, 12, 15, 50, 50, 50])]
    _run_script(ops, 64, 0)


def test_insert_batch_at_equals_insert_batch():
    """Continuing the insert from the matched node gives the same tree as inserting the whole
    prompt (slots, dup lengths, stamps through eviction order, node counts)."""
    rng = np.random.default_rng(21)
    for trial in range(20):
        t1, t2 = api.RadixTree(4096, trial), api.RadixTree(4096, trial)
        for rnd in range(6):
            prompts = [rng.integers(0, 3, size=rng.integers(1, 12)).astype(np.int32) for _ in range(8)]
            ind = np.concatenate([[0], np.cumsum([len(p) for p in prompts])])
            flat = np.concatenate(prompts)
            res = []
            for t in (t1, t2):
                ps, pind, last = t.match_prefix_batch(flat, ind)
                P = np.diff(pind)
                n_new = np.array([len(p) for p in prompts]) - P
                new = t.alloc_slots(int(n_new.sum()))
                res.append((ps, pind, last, P, n_new, new))
            (ps, pind, last, P, n_new, new) = res[0]
            assert np.array_equal(new, res[1][5]) and np.array_equal(last, res[1][2])
            nind = np.concatenate([[0], np.cumsum(n_new)])
            d1, l1 = t1.insert_batch_at(last, flat, ind, new, nind)
            full = np.empty(len(flat), np.int32)
            for b in range(len(prompts)):
                full[ind[b]:ind[b] + P[b]] = ps[pind[b]:pind[b + 1]]
                full[ind[b] + P[b]:ind[b + 1]] = new[nind[b]:nind[b + 1]]
            d2, l2 = t2.insert_batch(flat, ind, full)
            assert np.array_equal(d1, d2) and np.array_equal(l1, l2)
            for t, d in ((t1, d1), (t2, d2)):
                extra = [new[nind[b]:nind[b] + (d[b] - P[b])] for b in range(len(prompts)) if d[b] > P[b]]
                if extra:
                    t.free_slots(np.concatenate(extra))
            assert t1.stats() == t2.stats()
            t1.check()
            k = int(rng.integers(1, 20))
            assert t1.evict(k).tolist() == t2.evict(k).tolist()


def test_page_granular_matches_against_oracle():
    """With a page size p the tree reuses whole pages only: every match is the oracle's cached
    length cut down to a multiple of p, and inserts stay token granular."""
    for p in (2, 4, 16):
        rng = np.random.default_rng(30 + p)
        t = api.RadixTree(2048, p, page_size=p)
        m = PrefixCacheModel(2048, p)
        for _ in range(60):
            q = rng.integers(0, 3, size=int(rng.integers(1, 40))).astype(np.int32)
            want = m._cached_len(list(q))
            want -= want % p
            assert t.match_prefix_len(q) == want
            slots, k, _ = t.match_prefix(q)
            assert k == want
            k2, s2 = m.match(list(q)[:want])        # the oracle's match of the whole pages
            assert k2 == want and slots.tolist() == s2.tolist()
            if t.stats()["free_slots"] >= len(q):
                new = t.alloc_slots(len(q) - k)
                new2 = m.alloc.alloc(len(q) - k)
                assert new.tolist() == new2.tolist()
                d, _ = t.insert(q, np.concatenate([slots, new]))
                d2 = m.insert(list(q), np.concatenate([s2, new2]))
                assert d == d2 >= k
                t.free_slots(new[: d - k])          # the recomputed tail of the partial page
                m.alloc.release(new2[: d2 - k])
            if rng.random() < 0.2:
                k_ev = int(rng.integers(1, 20))
                assert t.evict(k_ev).tolist() == m.evict(k_ev).tolist()
            st = t.stats()
            assert st["cached_tokens"] == m.cached_tokens() and st["free_slots"] == len(m.alloc.free)
            t.check()
    with pytest.raises(api.RxError):
        api.radix_set_page_size(api.RadixTree(8, 0).h, 0)
