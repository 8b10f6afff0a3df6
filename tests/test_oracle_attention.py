"""Pins for the oracle's causal attention and merge (CPU only).

Each check is fixed by mathematics, not by re-running the oracle's own formula:
closed forms with hand-computed values, exact rational results, invariants, and the
split/merge identity.  A dropped scale, a wrong causal bound, a transposed operand or a
wrong query-head to kv-head map each fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention_rows, merge_states


def _one(q, k, v, pos, scale=1.0):
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    return attention_rows(q, np.asarray(pos, np.int64), k, v, scale)


def test_two_key_closed_form():
    # d=1, scale=1, q=1, k=(0, ln 2) -> weights (1/3, 2/3); v=(3, 6) -> o = 5, lse = ln 3.
    q = [[[1.0]]]
    k = [[[0.0]], [[math.log(2.0)]]]
    v = [[[3.0]], [[6.0]]]
    o, lse = _one(q, k, v, [1])
    assert abs(o[0, 0, 0] - 5.0) < 1e-6
    assert abs(lse[0, 0] - math.log(3.0)) < 1e-7
    # The same row at position 0 sees only the first key: o = v0 exactly, lse = 0.
    o, lse = _one(q, k, v, [0])
    assert o[0, 0, 0] == 3.0 and lse[0, 0] == 0.0


def test_dot_product_orientation():
    # q=(ln2, ln3), k0=e0, k1=e1 -> scores (ln2, ln3) -> weights (2/5, 3/5);
    # v0=(5,0), v1=(0,10) -> o=(2, 6).  Swapping q and k's roles or transposing K breaks it.
    q = [[[math.log(2.0), math.log(3.0)]]]
    k = [[[1.0, 0.0]], [[0.0, 1.0]]]
    v = [[[5.0, 0.0]], [[0.0, 10.0]]]
    o, lse = _one(q, k, v, [1])
    np.testing.assert_allclose(o[0, 0], [2.0, 6.0], rtol=0, atol=1e-6)
    assert abs(lse[0, 0] - math.log(5.0)) < 1e-7


def test_scale_is_applied():
    # scale 0.5: q=(2 ln 2, 0) -> scores (ln 2, 0) -> weights (2/3, 1/3); v0=(3,0), v1=(0,3) -> (2, 1).
    q = [[[2 * math.log(2.0), 0.0]]]
    k = [[[1.0, 0.0]], [[0.0, 1.0]]]
    v = [[[3.0, 0.0]], [[0.0, 3.0]]]
    o, _ = _one(q, k, v, [1], scale=0.5)
    np.testing.assert_allclose(o[0, 0], [2.0, 1.0], rtol=0, atol=1e-6)


def test_zero_scale_is_causal_mean_including_self():
    rng = np.random.default_rng(0)
    L, d = 9, 5
    k = rng.standard_normal((L, 1, d)).astype(np.float32)
    v = rng.standard_normal((L, 1, d)).astype(np.float32)
    q = rng.standard_normal((L, 1, d)).astype(np.float32)
    o, lse = attention_rows(q, np.arange(L), k, v, 0.0)
    for p in range(L):
        np.testing.assert_allclose(o[p, 0], v[: p + 1, 0].astype(np.float64).mean(0), rtol=0, atol=1e-6)
        assert abs(lse[p, 0] - math.log(p + 1)) < 1e-12


def test_gqa_contiguous_head_groups():
    # hq=6, hkv=3 (groups of 2): kv head g holds the constant value g+1 -> query head h gives h//2 + 1.
    L, d = 4, 3
    rng = np.random.default_rng(1)
    k = rng.standard_normal((L, 3, d)).astype(np.float32)
    v = np.zeros((L, 3, d), np.float32)
    for g in range(3):
        v[:, g, :] = g + 1
    q = rng.standard_normal((2, 6, d)).astype(np.float32)
    o, _ = attention_rows(q, np.array([1, 3]), k, v, 0.7)
    for h in range(6):
        np.testing.assert_allclose(o[:, h, :], h // 2 + 1, rtol=0, atol=1e-6)


def test_exact_rational_weights():
    # Scores ln(c_j) make the weights exactly c_j / sum(c): the exact answer is a fraction.
    rng = np.random.default_rng(2)
    L, hq, hkv = 7, 4, 2
    c = rng.integers(1, 9, size=(L, hkv))
    vals = rng.integers(-20, 21, size=(L, hkv))
    k = np.log(c).astype(np.float64)[:, :, None]          # d = 1, q = 1 -> score = ln c
    v = vals.astype(np.float32)[:, :, None]
    q = np.ones((L, hq, 1), np.float32)
    o, _ = attention_rows(q, np.arange(L), k.astype(np.float32), v, 1.0)
    kc = np.exp(k.astype(np.float32).astype(np.float64))[:, :, 0]   # weights of the stored keys
    for p in range(L):
        for h in range(hq):
            g = h // (hq // hkv)
            num = sum(Fraction(float(kc[j, g])) * int(vals[j, g]) for j in range(p + 1))
            den = sum(Fraction(float(kc[j, g])) for j in range(p + 1))
            assert abs(float(num / den) - o[p, h, 0]) < 1e-5


def test_hard_attention_limit():
    q = [[[1.0]]]
    k = [[[0.0]], [[0.0]], [[60.0]], [[0.0]]]
    v = [[[1.0]], [[2.0]], [[7.0]], [[4.0]]]
    o, lse = _one(q, k, v, [3])
    assert o[0, 0, 0] == 7.0 and abs(lse[0, 0] - 60.0) < 1e-12


def test_joint_key_permutation_invariance_for_full_row():
    rng = np.random.default_rng(3)
    L, d = 33, 16
    k = rng.standard_normal((L, 2, d)).astype(np.float32)
    v = rng.standard_normal((L, 2, d)).astype(np.float32)
    q = rng.standard_normal((1, 4, d)).astype(np.float32)
    perm = rng.permutation(L)
    o1, l1 = attention_rows(q, [L - 1], k, v, 0.25)
    o2, l2 = attention_rows(q, [L - 1], k[perm], v[perm], 0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-6)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)
    # Permuting V alone does change the answer (the pairing of k_j with v_j matters).
    o3, _ = attention_rows(q, [L - 1], k, v[perm], 0.25)
    assert np.abs(o3 - o1).max() > 1e-3


def test_split_merge_identity():
    # Softmax over a union of disjoint key sets equals the merge of the parts (in fp64).
    rng = np.random.default_rng(4)
    L, d = 50, 8
    k = rng.standard_normal((L, 1, d)).astype(np.float32)
    v = rng.standard_normal((L, 1, d)).astype(np.float32)
    q = rng.standard_normal((1, 2, d)).astype(np.float32)
    full_o, full_l = attention_rows(q, [L - 1], k, v, 0.3)
    cuts = [0, 7, 19, 20, 50]
    outs, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = attention_rows(q, [b - a - 1], k[a:b], v[a:b], 0.3)
        outs.append(o.astype(np.float64))
        lses.append(l)
    mo, ml = merge_states(outs, lses)
    np.testing.assert_allclose(mo, full_o, rtol=0, atol=2e-7)
    np.testing.assert_allclose(ml, full_l, rtol=0, atol=1e-12)


def test_merge_closed_form():
    # Two parts with lse ln 1 and ln 3 -> weights 1/4, 3/4.
    o, l = merge_states([[[4.0]], [[8.0]]], [[0.0], [math.log(3.0)]])
    assert abs(o[0, 0] - 7.0) < 1e-12 and abs(l[0] - math.log(4.0)) < 1e-12


def test_rejects_out_of_range_position():
    with pytest.raises(ValueError):
        _one([[[1.0]]], [[[0.0]]], [[[1.0]]], [1])
