"""Pins for the oracle's prefix-cache model, list matcher and slot allocator (CPU only)."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import ListMatcher, PrefixCacheModel, SlotAllocator, req_to_token, slot_order, splitmix64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_lcp(a, b):
    n = 0
    for x, y in zip(a, b):
        if x != y:
            break
        n += 1
    return n


def test_splitmix64_published_vector():
    lines = [l for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) if not l.startswith("#")]
    seed = int(lines[0].split()[1])
    want = [int(x) for x in lines[1:6]]
    got = [int(x) for x in splitmix64(seed, np.arange(1, 6))]
    assert got == want


def test_slot_order_is_a_permutation_and_seeded():
    o = slot_order(1000, 7)
    assert sorted(o.tolist()) == list(range(1000))
    assert not np.array_equal(o, np.arange(1000))
    assert np.array_equal(o, slot_order(1000, 7))
    assert not np.array_equal(o, slot_order(1000, 8))


def test_allocator_fifo_and_double_free():
    a = SlotAllocator(10, 3)
    order = slot_order(10, 3).tolist()
    s = a.alloc(4)
    assert s.tolist() == order[:4]
    assert a.alloc(7) is None                 # only 6 left: nothing allocated
    assert a.release([s[1], s[0]])
    assert a.alloc(6).tolist() == order[4:]
    assert a.alloc(2).tolist() == [s[1], s[0]]  # freed slots come back in release order
    assert not a.release([s[2], s[2]])        # duplicate in one call
    assert a.release([s[2]])
    assert not a.release([s[2]])              # already free


def test_req_to_token_layout():
    t = req_to_token([[5, 6], []], [[1], [2, 3, 4]], 5)
    assert t.tolist() == [[5, 6, 1, -1, -1], [2, 3, 4, -1, -1]]


@pytest.mark.parametrize("vocab", [2, 3, 4])
def test_model_match_equals_brute_force_lcp(vocab):
    rng = np.random.default_rng(vocab)
    for trial in range(40):
        m = PrefixCacheModel(4096, trial)
        inserted = []
        for step in range(12):
            seq = rng.integers(0, vocab, size=rng.integers(1, 11)).tolist()
            if rng.random() < 0.5:
                n, slots = m.match(seq)
                best = max([brute_lcp(seq, s) for s, _ in inserted], default=0)
                assert n == best
                # slots agree with every stored record on the matched part
                for s, sl in inserted:
                    l = brute_lcp(seq, s)
                    assert slots[:l].tolist() == sl[:l]
            else:
                n0 = max([brute_lcp(seq, s) for s, _ in inserted], default=0)
                new = m.alloc.alloc(len(seq))
                dup = m.insert(seq, new)
                assert dup == n0
                m.alloc.release(new[:dup])
                # the slots now cached for seq: old ones on the shared part, new after it
                _, cached = m.match(seq)
                inserted.append((seq, cached.tolist()))
            assert m.check_stamps_uniform()
            assert m.cached_tokens() + len(m.alloc.free) == 4096


def test_list_matcher_equals_brute_force():
    rng = np.random.default_rng(11)
    lm = ListMatcher()
    recs = []
    for _ in range(30):
        s = rng.integers(0, 3, size=rng.integers(1, 9)).tolist()
        sl = rng.integers(0, 1000, size=len(s)).tolist()
        lm.add(s, sl)
        recs.append((s, sl))
    for _ in range(200):
        q = rng.integers(0, 3, size=rng.integers(0, 10)).tolist()
        n, _ = lm.match(q)
        assert n == max([brute_lcp(q, s) for s, _ in recs], default=0)


def test_node_structure_split_and_count():
    m = PrefixCacheModel(64, 0)
    m.insert([1, 2, 3, 4], m.alloc.alloc(4))
    assert len(m.nodes()) == 1
    n, _ = m.match([1, 2, 9])              # match ends inside the edge: split at 2
    assert n == 2 and len(m.nodes()) == 2
    dup = m.insert([1, 2, 3, 7], m.alloc.alloc(4))
    assert dup == 3 and len(m.nodes()) == 4   # [1,2] [3] [4] [7]
    dup = m.insert([1, 2, 3, 4], m.alloc.alloc(4))
    assert dup == 4 and len(m.nodes()) == 4


def test_lru_eviction_order_and_locks():
    m = PrefixCacheModel(64, 0)
    a = m.alloc.alloc(3)
    m.insert([1, 1, 1], a)                  # clock 1
    b = m.alloc.alloc(3)
    m.insert([2, 2, 2], b)                  # clock 2
    c = m.alloc.alloc(3)
    m.insert([3, 3, 3], c)                  # clock 3
    m.match([1, 1, 1])                      # clock 4: [1,1,1] becomes most recent
    m.lock([2, 2, 2], 3)
    freed = m.evict(1)                      # LRU unlocked leaf: [3,3,3]
    assert freed.tolist() == c.tolist()
    freed = m.evict(1)                      # [2,2,2] is locked -> [1,1,1]
    assert freed.tolist() == a.tolist()
    assert m.evict(1).tolist() == []        # only the locked node is left
    m.lock([2, 2, 2], 3, -1)
    assert m.evict(10).tolist() == b.tolist()
    assert m.cached_tokens() == 0 and len(m.alloc.free) == 64


def test_evict_whole_leaves_then_parent():
    m = PrefixCacheModel(64, 0)
    m.insert([5, 6, 7], m.alloc.alloc(3))
    m.insert([5, 6, 8, 9], m.alloc.alloc(4))   # dup 2; leaves [7] and [8,9] under [5,6]
    freed = m.evict(1)
    assert len(freed) == 1                      # leaf [7] (older stamp) is one token
    freed = m.evict(2)                          # leaf [8,9] (2 tokens) is enough
    assert len(freed) == 2 and m.cached_tokens() == 2
    freed = m.evict(1)                          # now [5,6] is a leaf
    assert len(freed) == 2 and m.cached_tokens() == 0


def serve(m, prompt, n_out, out_tok):
    """The walk-through's serving flow: match the prompt, make room by evicting LRU leaves
    if the pool is short, allocate slots for the uncached tokens, insert prompt + reply."""
    full = list(prompt) + [out_tok] * n_out
    hit, _ = m.match(full)
    need = len(full) - hit
    short = need - len(m.alloc.free)
    evicted = m.evict(short) if short > 0 else np.zeros(0, np.int32)
    slots = m.alloc.alloc(need)
    assert slots is not None
    # matched positions keep their cached slots: the values passed for them are unused
    dup = m.insert(full, np.concatenate([np.full(hit, -1, np.int32), slots]))
    assert dup == hit
    return hit, evicted


def test_nine_step_walkthrough():
    spec = json.load(open(os.path.join(GOLDEN, "radix_walkthrough.json")))
    assert len(spec["steps"]) == 9
    SYS = [1, 2, 3, 4]
    m = PrefixCacheModel(64, 0)
    held = []

    def squeeze():            # other work holds every free slot: memory pressure
        if m.alloc.free:
            held.append(m.alloc.alloc(len(m.alloc.free)))

    def relax():
        for h in held:
            m.alloc.release(h)
        held.clear()

    cached = m._cached_len    # non-stamping lookup for the checks
    # step 1
    assert len(m.nodes()) == 0
    # step 2: one edge from the root
    serve(m, SYS + [10, 11], 2, 12)
    assert len(m.nodes()) == 1
    turn1 = SYS + [10, 11, 12, 12]
    # step 3: first session, second turn reuses the first turn
    hit, _ = serve(m, turn1 + [13], 2, 14)
    assert hit == len(turn1) and len(m.nodes()) == 2
    s1 = turn1 + [13, 14, 14]
    # step 4: second session shares only the system prompt: the step-3 path is split
    hit, _ = serve(m, SYS + [20, 21], 2, 22)
    assert hit == len(SYS) and len(m.nodes()) == 4
    s2 = SYS + [20, 21, 22, 22]
    # step 5: second session continues under memory pressure: the LRU leaf (the first
    # session's second turn) is evicted; the new turn hangs under the step-4 leaf.
    squeeze()
    hit, ev = serve(m, s2 + [23], 2, 24)
    assert hit == len(s2) and len(ev) == 3
    assert cached(s1) == len(turn1) and cached(s2 + [23, 24, 24]) == len(s2) + 3
    # step 6: few-shot query with a new first token: a new branch at the root
    relax()
    roots_before = m.nchild[()]
    serve(m, [30, 31, 32, 33, 34, 35], 1, 36)
    assert m.nchild[()] == roots_before + 1
    # step 7: more few-shot queries sharing the examples [30..34]: the step-6 node is split
    for q in (40, 41):
        hit, _ = serve(m, [30, 31, 32, 33, 34, q], 1, 36)
        assert hit == 5
    assert m.node_of((30, 31, 32, 33, 34))[-1] == (30, 31, 32, 33, 34)
    # step 8: the first session speaks again under pressure: every node of the second
    # session is evicted as least recently used, nothing else
    squeeze()
    few_shot_before = cached([30, 31, 32, 33, 34, 35, 36])
    hit, ev = serve(m, turn1 + [15], 3, 16)
    assert hit == len(turn1)
    assert cached(s2) == len(SYS) and len(ev) == 7
    assert cached([30, 31, 32, 33, 34, 35, 36]) == few_shot_before
    # step 9: more samples for the step-8 question: some nodes are evicted to make room
    total_ev = 0
    for sample in (50, 51, 52):
        squeeze()
        hit, ev = serve(m, turn1 + [15], 3, sample)
        assert hit == len(turn1) + 1
        total_ev += len(ev)
    assert total_ev > 0
    assert m.check_stamps_uniform()


def test_exhaustive_small_scripts_keep_invariants():
    # Every insert/match/evict interleaving over a 2-token vocabulary and short sequences.
    seqs = [list(s) for L in range(1, 4) for s in itertools.product([0, 1], repeat=L)]
    rng = np.random.default_rng(5)
    for trial in range(60):
        m = PrefixCacheModel(32, trial)
        for _ in range(10):
            op = rng.integers(0, 3)
            s = seqs[rng.integers(len(seqs))]
            if op == 0:
                m.match(s)
            elif op == 1:
                new = m.alloc.alloc(len(s))
                if new is None:
                    continue
                dup = m.insert(s, new)
                m.alloc.release(new[:dup])
            else:
                m.evict(int(rng.integers(1, 4)))
            assert m.check_stamps_uniform()
            assert m.cached_tokens() + len(m.alloc.free) == 32


def test_shared_groups_hand_worked():
    """Groups by first token, common length = longest common prefix (worked by hand)."""
    from oracle import shared_groups
    shared = list(range(100, 140))
    matched = [shared + [1000 + i] for i in range(5)] + [[9, 9, 9, 9]] + [shared[:10] + [55]] + [[]]
    gof, glen = shared_groups(matched, 1)
    assert gof.tolist() == [0, 0, 0, 0, 0, -1, 0, -1] and glen.tolist() == [10]
    gof, glen = shared_groups(matched[:5], 1)
    assert gof.tolist() == [0] * 5 and glen.tolist() == [40]
    gof, glen = shared_groups(matched[:5], 41)
    assert gof.tolist() == [-1] * 5 and glen.tolist() == []
    # two separate groups, numbered in order of first appearance; a prefix of another counts
    gof, glen = shared_groups([[5, 6, 7], [1, 2], [5, 6], [1, 2, 3], [8]], 1)
    assert gof.tolist() == [0, 1, 0, 1, -1] and glen.tolist() == [2, 2]
