"""GPU parity at the five workloads' full sizes.  The per-operation path (plan, upload, write,
attention) is compared in full at c1-c4 and on sampled rows at c5.  The path the benchmark
times -- PrefixCacheEngine.step (rx_step_plan + rx_step_launch) with cross-step overlap,
"auto" shared-prefix grouping, back-to-back steps on alternating device rows, and the
host-buffer pipeline of request ranges -- is compared at c3 in full and at c5 on a fixed
sample: all 64 heads, rows {0, 127, 128, 511, 1023} plus 27 seeded random rows of every
request, and every row of requests 0 and 31."""
import copy

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_cases import TOL_LSE, compare, expected_slots, oracle_rows, run_step, to_host_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_cached_kv_radix_gb300 import api
    api.load()


def _check_rows(w, out, lse, rows_of):
    got = to_host_f32(out)
    gl = lse.cpu().numpy()
    qo = w.qo_indptr()
    for b in range(w.batch):
        idx = rows_of(b)
        want, wl = oracle_rows(w, b, idx)
        sel = qo[b] + (np.arange(w.spec.req_new[b]) if idx is None else np.asarray(idx))
        compare(got[sel], want, f"{w.spec.name} request {b}")
        assert np.abs(gl[sel] - wl).max() <= TOL_LSE


def _check_table(w, plan, dev):
    pre, new, P = expected_slots(w)
    assert np.array_equal(plan.prefix_lens, P)
    r2t = dev["r2t"].cpu().numpy()
    for b in range(w.batch):
        row = np.concatenate([pre[b], new[b]])
        assert np.array_equal(r2t[b, :len(row)], row)
        assert (r2t[b, len(row):] == -1).all()


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_extend_full(name):
    w = W.generate(W.config(name))
    eng, plan, dev, out, lse, _ = run_step(w)
    assert eng.device_status() == 0
    _check_table(w, plan, dev)
    _check_rows(w, out, lse, lambda b: None)


def test_decode_c4_full():
    w = W.generate(W.config("c4"))
    eng, plan, dev, out, lse, grp = run_step(w, groups=True)
    assert eng.device_status() == 0
    assert grp is not None and grp.num_groups == 1 and grp.max_group_len == 4096
    _check_table(w, plan, dev)
    _check_rows(w, out, lse, lambda b: None)


def test_extend_c5_sampled():
    spec = W.config("c5")
    w = W.generate(spec)
    eng, plan, dev, out, lse, _ = run_step(w)
    assert eng.device_status() == 0
    _check_table(w, plan, dev)
    rng = np.random.default_rng(55)
    fixed = [0, 127, 128, 511, 1023]

    def rows(b):
        extra = rng.choice(np.setdiff1d(np.arange(1024), fixed), size=11, replace=False)
        return np.sort(np.concatenate([fixed, extra]))
    _check_rows(w, out, lse, rows)
    check_convex_bound(w, out)


def check_convex_bound(w, out):
    """A property of every row at any size: each output is a convex combination of its
    context's value rows, so per (head, dim) |o| <= max over the context of |v| (up to the
    bf16 rounding of P and of o, 2^-7 relative); every output is finite."""
    s = w.spec
    o = out.float()
    assert torch.isfinite(o).all()
    qo = w.qo_indptr()
    G = s.hq // s.hkv
    for b in range(w.batch):
        _, v = w.request_kv(b)
        vmax = np.abs(W.bf16_bits_to_f32(v) if s.dtype == "bf16" else v).max(axis=0)      # [hkv, d]
        bound = torch.from_numpy(np.repeat(vmax, G, axis=0) * (1 + 2.0 ** -7)).to(o.device)   # [hq, d]
        assert (o[qo[b]:qo[b + 1]].abs() <= bound).all(), f"request {b}: |o| above its context's max |v|"


# ---------------------------------------------------------------- the benchmark's one-call path
def _fresh_rows(w, seed):
    """A copy of workload w whose new tokens' q, k, v are fresh seeded draws (same shapes and
    distribution), for a second step on other device rows."""
    s = w.spec
    w2 = copy.copy(w)
    rng = np.random.default_rng([s.seed, 4242, seed])

    def draw(shape):
        x = rng.standard_normal(shape, dtype=np.float32)
        return W.f32_to_bf16_bits(x).reshape(shape) if s.dtype == "bf16" else x
    w2.req_q = [draw(x.shape) for x in w.req_q]
    w2.req_k = [draw(x.shape) for x in w.req_k]
    w2.req_v = [draw(x.shape) for x in w.req_v]
    return w2


def _check_plan(plan, w, pre, new_expected, P):
    assert np.array_equal(plan.prefix_lens, P), "match lengths differ from the oracle"
    for b in range(w.batch):
        assert np.array_equal(plan.prefix_slots[plan.prefix_indptr[b]:plan.prefix_indptr[b + 1]], pre[b])
    assert np.array_equal(plan.new_slots, new_expected), "new slots differ from the oracle allocator"


def _check_sampled(w, out, lse, rows_of, what):
    got = to_host_f32(out)
    gl = lse.cpu().numpy()
    qo = w.qo_indptr()
    for b in range(w.batch):
        idx = rows_of(b)
        want, wl = oracle_rows(w, b, idx)
        sel = qo[b] + (np.arange(w.spec.req_new[b]) if idx is None else np.asarray(idx))
        compare(got[sel], want, f"{what} request {b}")
        assert np.abs(gl[sel] - wl).max() <= TOL_LSE, f"{what} request {b}: lse"


def c5_sample(w, seed=55):
    """The c5 sample: rows {0, 127, 128, 511, 1023} plus 27 seeded random rows of every
    request (32 rows each, all heads), and every row of requests 0 and 31."""
    rng = np.random.default_rng(seed)
    fixed = np.array([0, 127, 128, 511, 1023])
    rows = {}
    for b in range(w.batch):
        n = w.spec.req_new[b]
        if b in (0, w.batch - 1):
            rows[b] = None
        else:
            extra = rng.choice(np.setdiff1d(np.arange(n), fixed), size=27, replace=False)
            rows[b] = np.sort(np.concatenate([fixed, extra]))
    return rows.get


@pytest.mark.parametrize("name", ["c3", "c5"])
def test_benchmark_path_matches_oracle(name):
    """The benchmark's step at full size, three ways: (A) device rows, overlap, groups "auto";
    (B) right after A with no synchronize, on a second set of device rows holding other values
    (its index-array copy runs under A's kernels); (C) host-buffer mode with four request ranges
    and overlap, on A's rows; (D) the same with the library's automatic ranges, as the benchmark
    runs it.  Every step has fresh new-token ids, inserts them and evicts as many tokens, as in
    the benchmark.  Slots are the oracle's bit for bit; A and B match the oracle (c3: every row;
    c5: the fixed sample for A, eight rows per request for B); C and D equal A bit for bit."""
    import bench
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine, _dev_from_host
    spec = W.config(name)
    w = W.generate(spec)
    s = spec
    eng = PrefixCacheEngine(s.dtype, s.hq, s.hkv, s.d, s.num_slots, s.seed)
    for i in range(len(s.histories)):
        k, v = w.history_kv(i)
        eng.populate(w.history_tokens(i), k, v)
    T = w.total_new()
    n_new = np.asarray(s.req_new, np.int64)
    used = {}
    inputs = []
    for j in range(4):
        prompts = bench.fresh_prompts(w, j, used)
        ind = np.concatenate([[0], np.cumsum([len(x) for x in prompts])]).astype(np.int64)
        inputs.append((np.concatenate(prompts).astype(np.int32), ind))
    w2 = _fresh_rows(w, 1)
    rows_a = [_dev_from_host(x, s.dtype, eng.device) for x in w.stacked_new()]
    rows_b = [_dev_from_host(x, s.dtype, eng.device) for x in w2.stacked_new()]
    outs = [torch.full_like(rows_a[0], float("nan")) for _ in range(2)]
    lses = [torch.full((T, s.hq), float("nan"), dtype=torch.float32, device=eng.device) for _ in range(2)]
    pre, new_a, P = expected_slots(w)
    plans = []
    for j, rows in enumerate((rows_a, rows_b)):     # A then B, no synchronize between them
        toks, ind = inputs[j]
        plans.append(eng.step(toks, ind, n_new, *rows, outs[j], lses[j], groups="auto", evict_tokens=T,
                              overlap=True))
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    eng.tree.check()
    want_new = step_slots(s, w, 4)
    assert np.array_equal(np.concatenate(new_a), want_new[0])
    for j in range(2):          # both plans' index arrays stay readable until the plan after next
        _check_plan(plans[j], w, pre, want_new[j], P)
    if name == "c3":
        _check_sampled(w, outs[0], lses[0], lambda b: None, f"{name} step A")
        _check_sampled(w2, outs[1], lses[1], lambda b: None, f"{name} step B")
    else:
        _check_sampled(w, outs[0], lses[0], c5_sample(w), f"{name} step A")
        check_convex_bound(w, outs[0])
        check_convex_bound(w2, outs[1])
        rng = np.random.default_rng(56)
        rows_b_of = {b: np.sort(np.concatenate([[0, 1023], rng.choice(np.arange(1, 1023), 6, replace=False)]))
                     for b in range(w.batch)}
        _check_sampled(w2, outs[1], lses[1], rows_b_of.get, f"{name} step B")
    # (C) host buffers, four request ranges, overlap; A's rows from pinned host memory; (D) the
    # same with the automatic ranges (a short last range of its own)
    host = [x.cpu().pin_memory() for x in rows_a]
    dev_rows = [torch.zeros_like(x) for x in rows_a]
    out_c = torch.empty_like(outs[0])
    lse_c = torch.empty_like(lses[0])
    for j, chunks in ((2, 4), (3, 0)):
        for x in dev_rows:
            x.zero_()                               # the library must fill them from the host copies
        torch.cuda.synchronize()                    # (with overlap the copies do not wait for this)
        out_h = torch.full(out_c.shape, float("nan"), dtype=out_c.dtype).pin_memory()
        lse_h = torch.full(lse_c.shape, float("nan"), dtype=torch.float32).pin_memory()
        toks, ind = inputs[j]
        plan_c = eng.step(toks, ind, n_new, *dev_rows, out_c, lse_c, groups="auto", evict_tokens=T,
                          host=(*host, out_h, lse_h), chunks=chunks, overlap=True)
        torch.cuda.synchronize()
        assert eng.device_status() == 0
        eng.tree.check()
        _check_plan(plan_c, w, pre, want_new[j], P)
        assert np.array_equal(out_h.view(torch.int16).numpy(), outs[0].view(torch.int16).cpu().numpy()), \
            f"host-buffer step (chunks={chunks}) differs from the device-row step"
        assert np.array_equal(lse_h.numpy(), lses[0].cpu().numpy())


def step_slots(s, w, k):
    """The oracle allocator's slots for each of k steps of T new tokens after the histories (the
    free list is far longer than what the steps take, so the slots that eviction returns to its
    tail are not reached)."""
    alloc = oracle.SlotAllocator(s.num_slots, s.seed)
    lm = oracle.ListMatcher()
    for i in range(len(s.histories)):
        toks = w.history_tokens(i)
        m, _ = lm.match(toks)
        alloc.alloc(len(toks) - m)
        lm.add(toks, np.zeros(len(toks), np.int32))
    T = w.total_new()
    return [alloc.alloc(T) for _ in range(k)]
