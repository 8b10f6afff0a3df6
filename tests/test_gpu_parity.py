"""GPU parity: the CUDA path through the C ABI against the oracle, element by element.

Small and medium cases that span several tiles and ragged tails, plus edge cases.
Slot tables are bit-exact; attention is within max-abs 2e-2, mean-abs 2e-3, relative
Frobenius 1e-2 per head, and log-sum-exp within 1e-3.
"""
import time

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_cases import (TOL_LSE, TOL_MAX_ABS, compare, expected_slots, f32, oracle_rows, run_step, to_host_f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_cached_kv_radix_gb300 import api
    api.load()


def check_tables(w, eng, plan, dev):
    pre, new, P = expected_slots(w)
    assert np.array_equal(plan.prefix_lens, P), "match lengths differ from the oracle"
    r2t = dev["r2t"].cpu().numpy()
    for b in range(w.batch):
        row = np.concatenate([pre[b], new[b]])
        assert np.array_equal(r2t[b, :len(row)], row), f"slot table row {b}"
        assert (r2t[b, len(row):] == -1).all()
    # new K/V rows landed bit-exactly at their slots
    q, kn, vn = w.stacked_new()
    allnew = np.concatenate(new) if len(new) else np.zeros(0, np.int32)
    if len(allnew):
        kp = eng.k_pool[torch.from_numpy(allnew.astype(np.int64)).cuda()].cpu()
        vp = eng.v_pool[torch.from_numpy(allnew.astype(np.int64)).cuda()].cpu()
        if w.spec.dtype == "bf16":
            assert np.array_equal(kp.view(torch.int16).numpy().view(np.uint16), kn)
            assert np.array_equal(vp.view(torch.int16).numpy().view(np.uint16), vn)
        else:
            assert np.array_equal(kp.numpy(), kn) and np.array_equal(vp.numpy(), vn)


def check_attention(w, out, lse, rows=None, max_abs=TOL_MAX_ABS):
    got = to_host_f32(out)
    got_lse = lse.cpu().numpy() if lse is not None else None
    qo = w.qo_indptr()
    for b in range(w.batch):
        if w.spec.req_new[b] == 0:
            continue
        idx = None if rows is None else rows[b]
        want, wl = oracle_rows(w, b, idx)
        sel = np.arange(qo[b], qo[b + 1]) if idx is None else qo[b] + np.asarray(idx)
        compare(got[sel], want, f"request {b}", max_abs)
        if got_lse is not None:
            assert np.abs(got_lse[sel] - wl).max() <= TOL_LSE, f"request {b}: lse"


def run_and_check(spec, groups=False, workload=None, max_abs=TOL_MAX_ABS):
    w = workload if workload is not None else W.generate(spec)
    eng, plan, dev, out, lse, _ = run_step(w, groups=groups)
    assert eng.device_status() == 0
    check_tables(w, eng, plan, dev)
    check_attention(w, out, lse, max_abs=max_abs)
    eng.tree.check()
    return w, eng


# ---------------------------------------------------------------- extend
def test_extend_c1_fp32():
    run_and_check(W.config("c1"))


def test_extend_c2_bf16_mha_d64():
    run_and_check(W.config("c2"))


def test_extend_gqa4_d128_ragged():
    # root 300 -> child 77; requests: full path + 130 new, half the root + 200 new (split),
    # no prefix + 37 new, full path + 1 new, root + 0 new tokens
    spec = W.Spec("gqa4-ragged", "bf16", 32, 8, 128, 1 << 14, W.QWEN_VOCAB, 11,
                  seg_parent=[-1, 0], seg_len=[300, 77], histories=[1],
                  req_seg=[1, 0, 0, 1, 0], req_cached=[377, 150, 0, 377, 300], req_new=[130, 200, 37, 1, 0])
    run_and_check(spec)


@pytest.mark.parametrize("hq,hkv", [(12, 4), (32, 2)])
def test_extend_group_sizes(hq, hkv):
    # 3 query heads per kv head do not tile 128 packed rows by whole tokens, so every Q and
    # output tile goes row by row; 16 per kv head make TMA boxes of 16 heads x 8 tokens.
    # Full tiles, a ragged last tile beside a full one, and a single token per request.
    spec = W.Spec(f"group{hq // hkv}", "bf16", hq, hkv, 128, 1 << 14, W.QWEN_VOCAB, 19,
                  seg_parent=[-1, 0], seg_len=[257, 64], histories=[1],
                  req_seg=[1, 0, 1], req_cached=[321, 100, 321], req_new=[150, 64, 1])
    run_and_check(spec)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4)])
def test_extend_d64_tensor_core_tiles(hq, hkv):
    # head dim 64 on the tcgen05 kernel (more than 8 rows per request and kv head): one TMA box
    # per tile row (64 columns), 1 or 2 query heads per kv head; full tiles beside ragged ones
    spec = W.Spec(f"d64-g{hq // hkv}", "bf16", hq, hkv, 64, 1 << 13, W.QWEN_VOCAB, 21,
                  seg_parent=[-1, 0], seg_len=[200, 90], histories=[1],
                  req_seg=[1, 0, 1], req_cached=[290, 57, 0], req_new=[256, 130, 41])
    run_and_check(spec)


def test_extend_gqa8_d128_many_tiles():
    spec = W.spec_multiturn("gqa8", "bf16", 64, 8, 128, 1 << 14, W.QWEN_VOCAB, 12, branches=2, branch_len=1200,
                            hit_len=1000, n_new=100)
    run_and_check(spec)


def test_extend_gqa4_d64():
    spec = W.spec_branching("gqa4-d64", "bf16", 16, 4, 64, 1 << 13, W.QWEN_VOCAB, 13, root=190, n_children=3,
                            child_len=45, leaves_per_child=2, n_new=70)
    run_and_check(spec)


def test_extend_without_cache_is_plain_causal_prefill():
    spec = W.Spec("nocache", "bf16", 8, 8, 128, 4096, W.QWEN_VOCAB, 14, seg_parent=[-1], seg_len=[5],
                  histories=[0], req_seg=[0, 0], req_cached=[0, 0], req_new=[333, 64])
    run_and_check(spec)


def test_extend_fp32_gqa():
    spec = W.spec_branching("f32-gqa", "f32", 8, 2, 128, 2048, W.QWEN_VOCAB, 15, root=100, n_children=2,
                            child_len=20, leaves_per_child=2, n_new=9)
    run_and_check(spec)


def grow_keys(w, rate):
    """Scale every key by 1 + rate * (its position in the context), in place: later key tiles
    raise the running row max by more than the lazy-rescale threshold again and again, so the
    kernels' rescale of the partial output (after the previous PV has completed) runs often.
    Position = offset along the segment path for cached keys, P_b + i for new ones."""
    s = w.spec
    start = {}
    for seg in range(len(s.seg_parent)):
        path = w.seg_path(seg)
        start[seg] = sum(s.seg_len[x] for x in path[:-1])
    def scaled(a, p0):
        f = f32(a, s.dtype) * (1.0 + rate * (p0 + np.arange(len(a), dtype=np.float32)))[:, None, None]
        return W.f32_to_bf16_bits(f) if s.dtype == "bf16" else f.astype(np.float32)
    w.seg_k = [scaled(k, start[i]) for i, k in enumerate(w.seg_k)]
    w.req_k = [scaled(k, s.req_cached[b]) for b, k in enumerate(w.req_k)]
    return w


def peaked_max_abs(w):
    """Max-abs bound when attention concentrates on single keys: P is rounded to bf16 before
    PV and the output to bf16 after it, each within 2^-8 relative, so a row that is nearly one
    value row v is off by up to about 2^-7 max|v| (mean-abs and relative bounds stay)."""
    vmax = max(np.abs(f32(v, w.spec.dtype)).max() for v in w.seg_v + w.req_v)
    return max(TOL_MAX_ABS, 2.0 ** -7 * vmax)


def test_extend_rescales_as_scores_grow():
    spec = W.spec_multiturn("grow", "bf16", 64, 8, 128, 1 << 14, W.QWEN_VOCAB, 16, branches=2, branch_len=1200,
                            hit_len=1000, n_new=100)
    w = grow_keys(W.generate(spec), 0.02)
    run_and_check(spec, workload=w, max_abs=peaked_max_abs(w))


# ---------------------------------------------------------------- decode
def small_decode(dtype="bf16", hq=32, hkv=8, d=128, seed=21):
    return W.spec_decode("dec-small", dtype, hq, hkv, d, 1 << 16, W.QWEN_VOCAB, seed, batch=24, share_frac=0.6,
                         shared_len=700, min_len=1, max_len=3000)


def test_decode_split_kv():
    run_and_check(small_decode())


def test_decode_shared_prefix_groups():
    w, eng = run_and_check(small_decode(), groups=True)


def test_decode_shared_prefix_groups_rescale():
    spec = small_decode(seed=26)
    w = grow_keys(W.generate(spec), 0.01)
    run_and_check(spec, groups=True, workload=w, max_abs=peaked_max_abs(w))


def test_decode_groups_equal_no_groups():
    spec = small_decode(seed=22)
    w = W.generate(spec)
    _, _, _, o1, l1, _ = run_step(w, groups=False)
    _, _, _, o2, l2, grp = run_step(w, groups=True)
    assert grp is not None and grp.num_groups >= 1
    a, b = to_host_f32(o1), to_host_f32(o2)
    assert np.abs(a - b).max() <= 1e-2
    assert np.abs(l1.cpu().numpy() - l2.cpu().numpy()).max() <= 1e-3


def test_decode_mha_d64():
    run_and_check(small_decode(hq=12, hkv=12, d=64, seed=23))


def test_decode_fp32():
    run_and_check(W.spec_decode("dec-f32", "f32", 8, 2, 64, 8192, W.QWEN_VOCAB, 24, batch=6, share_frac=0.5,
                                shared_len=50, min_len=1, max_len=300))


def test_decode_length_one():
    spec = W.spec_decode("dec-one", "bf16", 32, 8, 128, 4096, W.QWEN_VOCAB, 25, batch=5, share_frac=0.0,
                         shared_len=10, min_len=1, max_len=1)
    run_and_check(spec)


# ---------------------------------------------------------------- edge cases and errors
def test_empty_batch_is_a_no_op():
    from prefix_cached_kv_radix_gb300 import api
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine
    eng = PrefixCacheEngine("bf16", 32, 8, 128, 1024, 1)
    z = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device="cuda")
    r2t = torch.zeros(1, 8, dtype=torch.int32, device="cuda")
    i64 = torch.zeros(1, dtype=torch.int64, device="cuda")
    i32 = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.prefix_extend_attention(eng.desc, 0, z, i64, i32, r2t, eng.k_pool, eng.v_pool, z, None, 1, eng.status)
    api.kv_pool_write(eng.desc, 0, i32, i64, i32, i64, z, z, eng.k_pool, eng.v_pool, r2t, 0, eng.status)
    torch.cuda.synchronize()
    assert eng.device_status() == 0


def _bad_table_case(kind):
    """A hand-built slot table with one out-of-range slot (or a length past the stride);
    the kernels' own bounds checks must turn it into a device status, not a fault."""
    from prefix_cached_kv_radix_gb300 import api
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine
    eng = PrefixCacheEngine("bf16", 8, 8, 128, 256, 2, poison=False)
    eng.k_pool.zero_()
    eng.v_pool.zero_()
    L = 40
    r2t = torch.arange(L, dtype=torch.int32, device="cuda").view(1, L)
    if kind == "slot":
        r2t[0, 17] = 256 + 5
    q = torch.randn(4, 8, 128, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    qo = torch.tensor([0, 4], dtype=torch.int64, device="cuda")
    P = torch.tensor([L - 4 if kind == "slot" else L], dtype=torch.int32, device="cuda")
    return api, eng, r2t, q, out, qo, P


def test_bad_slot_sets_status_extend():
    api, eng, r2t, q, out, qo, P = _bad_table_case("slot")
    api.prefix_extend_attention(eng.desc, 1, q, qo, P, r2t, eng.k_pool, eng.v_pool, out, None, 4, eng.status)
    torch.cuda.synchronize()
    assert eng.device_status() == api.RX_DEV_BAD_SLOT


def test_bad_length_sets_status_extend():
    api, eng, r2t, q, out, qo, P = _bad_table_case("length")
    api.prefix_extend_attention(eng.desc, 1, q, qo, P, r2t, eng.k_pool, eng.v_pool, out, None, 4, eng.status)
    torch.cuda.synchronize()
    assert eng.device_status() == api.RX_DEV_BAD_LENGTH


def test_bad_slot_sets_status_decode():
    api, eng, r2t, q, out, qo, P = _bad_table_case("slot")
    qd = q[:1].contiguous()
    od = torch.empty_like(qd)
    lens = torch.tensor([40], dtype=torch.int32, device="cuda")
    ws = torch.empty(api.decode_workspace_bytes(eng.desc, 1, 40), dtype=torch.uint8, device="cuda")
    api.decode_attention(eng.desc, 1, qd, r2t, lens, eng.k_pool, eng.v_pool, od, None, 40, ws, eng.status)
    torch.cuda.synchronize()
    assert eng.device_status() == api.RX_DEV_BAD_SLOT


def test_bounded_wait_times_out_and_device_stays_usable():
    """A kernel's bounded wait on a barrier that nothing arrives at gives up after its limit,
    records RX_DEV_TIMEOUT in the status word and ends; the device then runs a normal step."""
    from prefix_cached_kv_radix_gb300 import api
    api.load()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    api.rx_wait_selftest(status, 5_000_000)          # 5 ms
    torch.cuda.synchronize()
    assert int(status.item()) == api.RX_DEV_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # a second call leaves a recorded code in place
    api.rx_wait_selftest(status, 1_000)
    torch.cuda.synchronize()
    assert int(status.item()) == api.RX_DEV_TIMEOUT
    run_and_check(W.config("c1"))


def test_workspace_too_small_is_rejected_on_host():
    from prefix_cached_kv_radix_gb300 import api
    api_, eng, r2t, q, out, qo, P = _bad_table_case("length")
    lens = torch.tensor([40], dtype=torch.int32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.RxError):
        api.decode_attention(eng.desc, 1, q[:1].contiguous(), r2t, lens, eng.k_pool, eng.v_pool,
                             torch.empty_like(q[:1]), None, 40, ws, eng.status)


def test_step_then_evict_restores_cache():
    spec = W.config("c2")
    w = W.generate(spec)
    eng, plan, dev, out, lse, _ = run_step(w)
    before = eng.tree.stats()
    eng.commit(plan)
    after = eng.tree.stats()
    assert after["cached_tokens"] == before["cached_tokens"] + w.total_new()
    freed = eng.release(w.total_new())
    assert len(freed) == w.total_new() and sorted(freed.tolist()) == sorted(plan.new_slots.tolist())
    assert eng.tree.stats()["cached_tokens"] == before["cached_tokens"]
    eng.tree.check()
    # the same step again sees the same hits (the prefix stayed cached)
    plan2 = eng.plan([w.request_tokens(b) for b in range(w.batch)], spec.req_new)
    assert np.array_equal(plan2.prefix_lens, plan.prefix_lens)


# ---------------------------------------------------------------- grouped extend (shared prefix stacked)
def run_grouped(spec, groups="auto", expect_grouped=True):
    w = W.generate(spec)
    eng, plan, dev, out, lse, grp = run_step(w, groups=groups)
    assert eng.device_status() == 0
    assert (grp is not None) == expect_grouped
    check_tables(w, eng, plan, dev)
    check_attention(w, out, lse)
    return w, out, lse


def test_grouped_extend_c2():
    run_grouped(W.config("c2"), groups=True)


def test_auto_grouping_leaves_small_extend_ungrouped():
    # c2's 7-8 rows per (request, head) over 417 keys fit the small-extend kernel: "auto"
    # does not stack them, and the outputs are the oracle's either way
    run_grouped(W.config("c2"), groups="auto", expect_grouped=False)


def test_grouped_extend_private_cached_tails():
    # a shared 300-token root, 6 children of 40 tokens, 3 requests per child with 5 new tokens:
    # the group shares the root; each request's child tokens and own tokens are private
    spec = W.spec_branching("grp-tails", "bf16", 12, 12, 64, 1 << 14, W.GPT2_VOCAB, 41, root=300, n_children=6,
                            child_len=40, leaves_per_child=3, n_new=5)
    run_grouped(spec, groups=True)


def test_grouped_extend_gqa_d128():
    spec = W.spec_shared_prompt("grp-gqa", "bf16", 32, 8, 128, 1 << 14, W.QWEN_VOCAB, 42, 700, [3, 9, 1, 16, 7, 12])
    run_grouped(spec)


def test_grouped_extend_forced_with_ungrouped_requests():
    # two roots: requests under root A form a group, the single request on root B does not
    spec = W.Spec("grp-mixed", "bf16", 8, 2, 128, 1 << 13, W.QWEN_VOCAB, 43, seg_parent=[-1, -1],
                  seg_len=[260, 90], histories=[0, 1], req_seg=[0, 0, 0, 1], req_cached=[260, 260, 130, 90],
                  req_new=[4, 6, 3, 5])
    run_grouped(spec, groups=True)


def test_grouped_equals_ungrouped_extend():
    spec = W.config("c2")
    w = W.generate(spec)
    _, _, _, o1, l1, g1 = run_step(w, groups=False)
    _, _, _, o2, l2, g2 = run_step(w, groups=True)
    assert g1 is None and g2 is not None      # small-extend kernel vs the grouped path
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


# ---------------------------------------------------------------- page-granular reuse
@pytest.mark.parametrize("name,page", [("c2", 16), ("c1", 48), ("c2", 64)])
def test_page_granular_reuse_recomputes_the_partial_page(name, page):
    """With a page size the cached prefix is reused in whole pages only: the tail of the
    partly matched page is recomputed (its K/V written again to new slots, its rows
    attended) and the outputs of every computed row still equal the oracle's."""
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine, _dev_from_host
    import oracle
    spec = W.config(name)
    w = W.generate(spec)
    s = spec
    eng = PrefixCacheEngine(s.dtype, s.hq, s.hkv, s.d, s.num_slots, s.seed, page_size=page)
    for i in range(len(s.histories)):
        k, v = w.history_kv(i)
        eng.populate(w.history_tokens(i), k, v)
    prompts = [w.request_tokens(b) for b in range(w.batch)]
    n_new = eng.new_token_counts(prompts)
    P_r = np.array([len(p) for p in prompts]) - n_new
    assert (P_r % page == 0).all() and (P_r <= np.array(s.req_cached)).all()
    assert (P_r < np.array(s.req_cached)).any()          # some prefix tails are recomputed
    rng = np.random.default_rng(99)
    qs, ks, vs, rows = [], [], [], []
    for b in range(w.batch):
        kf, vf = w.request_kv(b)
        lo, P = int(P_r[b]), s.req_cached[b]
        extra_q = rng.standard_normal((P - lo, s.hq, s.d)).astype(np.float32)
        if s.dtype == "bf16":
            extra_q = W.f32_to_bf16_bits(extra_q)
        qs.append(np.concatenate([extra_q, w.req_q[b]]))
        ks.append(kf[lo:])
        vs.append(vf[lo:])
        rows.append((lo, qs[-1]))
    plan = eng.plan(prompts, n_new)
    assert np.array_equal(plan.prefix_lens, P_r)
    dev = eng.upload(plan)
    qd, kd, vd = (_dev_from_host(np.concatenate(x), s.dtype, eng.device) for x in (qs, ks, vs))
    out = torch.empty_like(qd)
    eng.write(plan, dev, kd, vd)
    eng.extend(plan, dev, qd, out, None)
    free_before = eng.tree.stats()["free_slots"]
    eng.finish(plan)
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    # the recomputed tail's new slots came back as duplicates
    assert eng.tree.stats()["free_slots"] - free_before == int((np.array(s.req_cached) - P_r).sum())
    got = to_host_f32(out)
    qo = np.concatenate([[0], np.cumsum(n_new)])
    for b in range(w.batch):
        kf, vf = w.request_kv(b)
        lo, qb = rows[b]
        want, _ = oracle.attention_rows(f32(qb, s.dtype), lo + np.arange(len(qb)), f32(kf, s.dtype),
                                        f32(vf, s.dtype), s.scale)
        compare(got[qo[b]:qo[b + 1]], want, f"{name} page {page} request {b}")
    eng.tree.check()


# ---------------------------------------------------------------- one-call step
@pytest.mark.parametrize("name", ["c1", "c2", "c4"])
def test_one_call_step_matches_oracle(name):
    """engine.step: rx_step_plan then rx_step_launch (copy, kv_pool_write, attention with the
    plan's groups, insert/evict/unpin) gives the oracle's slots and attention; a second step
    planned into the other staging buffer while the first may still run stays correct."""
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine, _dev_from_host
    spec = W.config(name)
    w = W.generate(spec)
    s = spec
    eng = PrefixCacheEngine(s.dtype, s.hq, s.hkv, s.d, s.num_slots, s.seed)
    for i in range(len(s.histories)):
        k, v = w.history_kv(i)
        eng.populate(w.history_tokens(i), k, v)
    prompts = [w.request_tokens(b) for b in range(w.batch)]
    ind = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
    toks = np.concatenate(prompts).astype(np.int32)
    q, kn, vn = w.stacked_new()
    qd, kd, vd = (_dev_from_host(x, s.dtype, eng.device) for x in (q, kn, vn))
    out = torch.empty_like(qd)
    lse = torch.empty(qd.shape[0], s.hq, dtype=torch.float32, device=eng.device)
    pre, new, P = expected_slots(w)
    plan = eng.step(toks, ind, s.req_new, qd, kd, vd, out, lse, decode=s.decode,
                    groups=True if s.decode else "auto")
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    assert np.array_equal(plan.prefix_lens, P)
    for b in range(w.batch):
        assert plan.prefix_slots[plan.prefix_indptr[b]:plan.prefix_indptr[b + 1]].tolist() == pre[b].tolist()
        assert plan.new_slots[plan.qo_indptr[b]:plan.qo_indptr[b + 1]].tolist() == new[b].tolist()
    got, got_lse = to_host_f32(out), lse.cpu().numpy()
    qo = np.concatenate([[0], np.cumsum(s.req_new)])
    for b in range(w.batch):
        want, want_lse = oracle_rows(w, b)
        compare(got[qo[b]:qo[b + 1]], want, f"{name} request {b}")
        assert np.abs(got_lse[qo[b]:qo[b + 1]] - want_lse).max() <= TOL_LSE
    # the step inserted its new tokens: the same prompts are now fully cached
    assert eng.new_token_counts(prompts).tolist() == [0] * w.batch
    eng.tree.check()


# ---------------------------------------------------------------- small extend (decode-shaped)
@pytest.mark.parametrize("hq,hkv,d,new_lens,prefix", [(32, 8, 128, [1, 2, 2, 1, 2, 1], 600),
                                                       (8, 8, 64, [8, 7, 3, 8, 1], 1000),
                                                       (16, 2, 128, [1, 1, 1], 37)])
def test_small_extend_rows(hq, hkv, d, new_lens, prefix):
    """A few new tokens per request (new tokens x heads per kv head <= 8) over at most 1024
    keys run on the decode-shaped kernel with per-row causal limits; every row equals the
    oracle's (ragged lengths, GQA, D 64 and 128, the 1024-key edge)."""
    spec = W.spec_shared_prompt("small", "bf16", hq, hkv, d, 8192, 50257, 17, prefix, new_lens)
    w = W.generate(spec)
    eng, plan, dev, out, lse, _ = run_step(w)
    assert plan.layout.num_groups == 0 and max(new_lens) * (hq // hkv) <= 8 and plan.stride <= 1024
    check_tables(w, eng, plan, dev)
    got, got_lse = to_host_f32(out), lse.cpu().numpy()
    qo = w.qo_indptr()
    for b in range(w.batch):
        want, want_lse = oracle_rows(w, b)
        compare(got[qo[b]:qo[b + 1]], want, f"small extend request {b}")
        assert np.abs(got_lse[qo[b]:qo[b + 1]] - want_lse).max() <= TOL_LSE


# ---------------------------------------------------------------- host-buffer step (e2e path)
def _engine_for(w):
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine
    s = w.spec
    eng = PrefixCacheEngine(s.dtype, s.hq, s.hkv, s.d, s.num_slots, s.seed)
    for i in range(len(s.histories)):
        k, v = w.history_kv(i)
        eng.populate(w.history_tokens(i), k, v)
    return eng


@pytest.mark.parametrize("chunks", [1, 3, 0])
def test_host_buffer_step_equals_device_step(chunks):
    """rx_step_launch in host-buffer mode (rows copied in and the output out by the library, as
    a pipeline of request ranges) gives exactly the device-buffer step's output and lse."""
    from prefix_cached_kv_radix_gb300.engine import _dev_from_host
    spec = W.Spec("gqa4-ragged-host", "bf16", 32, 8, 128, 1 << 14, W.QWEN_VOCAB, 31,
                  seg_parent=[-1, 0], seg_len=[300, 77], histories=[1],
                  req_seg=[1, 0, 0, 1, 0, 1], req_cached=[377, 150, 0, 377, 300, 200],
                  req_new=[130, 200, 37, 1, 0, 64])
    w = W.generate(spec)
    prompts = [w.request_tokens(b) for b in range(w.batch)]
    ind = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
    toks = np.concatenate(prompts).astype(np.int32)
    q, kn, vn = w.stacked_new()
    outs = []
    for host in (False, True):
        eng = _engine_for(w)
        qd, kd, vd = (_dev_from_host(x, spec.dtype, eng.device) for x in (q, kn, vn))
        out = torch.empty_like(qd)
        lse = torch.empty(qd.shape[0], spec.hq, dtype=torch.float32, device=eng.device)
        if host:
            hq_, hk_, hv_ = (x.cpu().pin_memory() for x in (qd, kd, vd))
            for x in (qd, kd, vd):
                x.zero_()                           # the library must fill them from the host copies
            out_h = torch.full(out.shape, float("nan"), dtype=out.dtype).pin_memory()
            lse_h = torch.full(lse.shape, float("nan"), dtype=torch.float32).pin_memory()
            eng.step(toks, ind, spec.req_new, qd, kd, vd, out, lse, host=(hq_, hk_, hv_, out_h, lse_h), chunks=chunks)
            torch.cuda.synchronize()
            outs.append((out_h.float().numpy(), lse_h.numpy()))
        else:
            eng.step(toks, ind, spec.req_new, qd, kd, vd, out, lse)
            torch.cuda.synchronize()
            outs.append((to_host_f32(out), lse.cpu().numpy()))
        assert eng.device_status() == 0
        eng.tree.check()
    (o_d, l_d), (o_h, l_h) = outs
    assert np.array_equal(o_d, o_h) and np.array_equal(l_d, l_h)
    qo = w.qo_indptr()
    for b in range(w.batch):
        if spec.req_new[b]:
            want, _ = oracle_rows(w, b)
            compare(o_h[qo[b]:qo[b + 1]], want, f"request {b}")


def test_host_buffer_automatic_ranges_end_with_an_empty_request():
    """The automatic range split on a step large enough for several ranges (147 MB of rows):
    the last eighth of the last range runs on its own, which here is a request with no new
    tokens (its range copies and computes nothing but still writes its slot-table row).  The
    host-buffer step equals the device-row step bit for bit, and sampled rows the oracle."""
    from prefix_cached_kv_radix_gb300.engine import _dev_from_host
    n = 800
    spec = W.Spec("gqa4-auto-ranges", "bf16", 32, 8, 128, 1 << 14, W.QWEN_VOCAB, 37,
                  seg_parent=[-1], seg_len=[300], histories=[0],
                  req_seg=[0] * 10, req_cached=[300, 0, 300, 120, 300, 0, 300, 300, 64, 300],
                  req_new=[n] * 9 + [0])
    w = W.generate(spec)
    prompts = [w.request_tokens(b) for b in range(w.batch)]
    ind = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
    toks = np.concatenate(prompts).astype(np.int32)
    q, kn, vn = w.stacked_new()
    outs = []
    for host in (False, True):
        eng = _engine_for(w)
        qd, kd, vd = (_dev_from_host(x, spec.dtype, eng.device) for x in (q, kn, vn))
        out = torch.empty_like(qd)
        lse = torch.empty(qd.shape[0], spec.hq, dtype=torch.float32, device=eng.device)
        if host:
            hq_, hk_, hv_ = (x.cpu().pin_memory() for x in (qd, kd, vd))
            for x in (qd, kd, vd):
                x.zero_()
            torch.cuda.synchronize()
            out_h = torch.full(out.shape, float("nan"), dtype=out.dtype).pin_memory()
            lse_h = torch.full(lse.shape, float("nan"), dtype=torch.float32).pin_memory()
            plan = eng.step(toks, ind, spec.req_new, qd, kd, vd, out, lse, host=(hq_, hk_, hv_, out_h, lse_h), chunks=0)
            torch.cuda.synchronize()
            outs.append((out_h.float().numpy(), lse_h.numpy()))
        else:
            plan = eng.step(toks, ind, spec.req_new, qd, kd, vd, out, lse)
            torch.cuda.synchronize()
            outs.append((to_host_f32(out), lse.cpu().numpy()))
        assert eng.device_status() == 0
        eng.tree.check()
        assert np.array_equal(plan.prefix_lens, np.asarray(spec.req_cached, np.int32))
    (o_d, l_d), (o_h, l_h) = outs
    assert np.array_equal(o_d, o_h) and np.array_equal(l_d, l_h)
    qo = w.qo_indptr()
    for b in (0, 3, 8):
        idx = np.array([0, 1, n // 2, n - 1])
        want, want_lse = oracle_rows(w, b, idx)
        compare(o_h[qo[b] + idx], want, f"request {b}")
        assert np.abs(l_h[qo[b] + idx] - want_lse).max() <= TOL_LSE


def test_host_buffer_steps_overlap_back_to_back():
    """Host-buffer steps back to back with overlap: two sets of device rows used in turn, each
    step's input copies waiting only for the kernels of the last step that read the same rows
    (so they run under the previous step's kernels), no synchronize between steps.  Every
    step's output equals, bit for bit, the same step run one at a time on device rows."""
    from prefix_cached_kv_radix_gb300.engine import _dev_from_host
    spec = W.Spec("gqa4-ragged-overlap", "bf16", 32, 8, 128, 1 << 14, W.QWEN_VOCAB, 33,
                  seg_parent=[-1, 0], seg_len=[300, 77], histories=[1],
                  req_seg=[1, 0, 0, 1, 0, 1], req_cached=[377, 150, 0, 377, 300, 200],
                  req_new=[130, 200, 37, 1, 0, 64])
    w = W.generate(spec)
    rng = np.random.default_rng(5)
    q, kn, vn = w.stacked_new()
    steps = []
    for j in range(4):   # fresh new tokens and different rows at every step
        prompts = [np.concatenate([w.request_prefix_tokens(b),
                                   rng.integers(1, spec.vocab, size=spec.req_new[b])]).astype(np.int32)
                   for b in range(w.batch)]
        ind = np.concatenate([[0], np.cumsum([len(x) for x in prompts])]).astype(np.int64)
        steps.append((np.concatenate(prompts).astype(np.int32), ind, 1.0 + 0.25 * j))
    ref = []
    eng = _engine_for(w)
    base = [_dev_from_host(x, spec.dtype, eng.device) for x in (q, kn, vn)]
    out = torch.empty_like(base[0])
    for toks, ind, sc in steps:
        rows = [x * sc for x in base]
        eng.step(toks, ind, spec.req_new, *rows, out)
        torch.cuda.synchronize()
        ref.append(to_host_f32(out))
    assert eng.device_status() == 0
    eng = _engine_for(w)
    sets = [[torch.zeros_like(x) for x in base] for _ in range(2)]
    out = torch.empty_like(base[0])
    host_rows = [[(x * sc).cpu().pin_memory() for x in base] for _, _, sc in steps]
    outs_h = [torch.full(out.shape, float("nan"), dtype=out.dtype).pin_memory() for _ in steps]
    for j, (toks, ind, _) in enumerate(steps):
        eng.step(toks, ind, spec.req_new, *sets[j % 2], out, host=(*host_rows[j], outs_h[j]), chunks=3,
                 overlap=True)
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    eng.tree.check()
    for j in range(len(steps)):
        assert np.array_equal(outs_h[j].float().numpy(), ref[j]), f"step {j}"


def test_device_steps_overlap_back_to_back():
    """Device-row steps back to back with overlap (the index arrays copied on a copy stream
    under the previous step's kernels, into the engine's two device staging buffers in turn),
    no synchronize between steps: every step's output equals, bit for bit, the same step run
    one at a time."""
    from prefix_cached_kv_radix_gb300.engine import _dev_from_host
    spec = W.Spec("gqa4-ragged-overlap-dev", "bf16", 32, 8, 128, 1 << 14, W.QWEN_VOCAB, 35,
                  seg_parent=[-1, 0], seg_len=[300, 77], histories=[1],
                  req_seg=[1, 0, 0, 1, 0, 1], req_cached=[377, 150, 0, 377, 300, 200],
                  req_new=[130, 200, 37, 1, 0, 64])
    w = W.generate(spec)
    rng = np.random.default_rng(6)
    q, kn, vn = w.stacked_new()
    steps = []
    for j in range(5):
        prompts = [np.concatenate([w.request_prefix_tokens(b),
                                   rng.integers(1, spec.vocab, size=spec.req_new[b])]).astype(np.int32)
                   for b in range(w.batch)]
        ind = np.concatenate([[0], np.cumsum([len(x) for x in prompts])]).astype(np.int64)
        steps.append((np.concatenate(prompts).astype(np.int32), ind, 1.0 + 0.25 * j))
    results = []
    for overlap in (False, True):
        eng = _engine_for(w)
        base = [_dev_from_host(x, spec.dtype, eng.device) for x in (q, kn, vn)]
        rows = [[x * sc for x in base] for _, _, sc in steps]
        outs = [torch.empty_like(base[0]) for _ in steps]
        for j, (toks, ind, _) in enumerate(steps):
            eng.step(toks, ind, spec.req_new, *rows[j], outs[j], overlap=overlap)
            if not overlap:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert eng.device_status() == 0
        eng.tree.check()
        results.append([to_host_f32(o) for o in outs])
    for j in range(len(steps)):
        assert np.array_equal(results[0][j], results[1][j]), f"step {j}"


@pytest.mark.gpu
def test_small_extend_steps_back_to_back():
    """Small-extend steps (a few rows per request and kv head: the small-extend kernel, launched
    behind kv_pool_write with programmatic serialization, the index arrays read by kv_pool_write
    through the staging buffer's mapping and the buffer's reuse signalled in host memory) run
    back to back with no synchronize: every step's output equals, bit for bit, the same step run
    one at a time, and the first equals the oracle."""
    from prefix_cached_kv_radix_gb300.engine import _dev_from_host
    spec = W.spec_shared_prompt("small-b2b", "bf16", 12, 12, 64, 1 << 14, W.GPT2_VOCAB, 41, 200,
                                [7, 8, 5, 8, 1, 6, 8, 3, 7, 2, 8, 4])
    w = W.generate(spec)
    rng = np.random.default_rng(9)
    q, kn, vn = w.stacked_new()
    steps = []
    for j in range(6):
        prompts = [np.concatenate([w.request_prefix_tokens(b),
                                   rng.integers(1, spec.vocab, size=spec.req_new[b])]).astype(np.int32)
                   for b in range(w.batch)]
        ind = np.concatenate([[0], np.cumsum([len(x) for x in prompts])]).astype(np.int64)
        steps.append((np.concatenate(prompts).astype(np.int32), ind, 1.0 + 0.25 * j))
    T = int(sum(spec.req_new))
    results = []
    for serial in (True, False):
        eng = _engine_for(w)
        base = [_dev_from_host(x, spec.dtype, eng.device) for x in (q, kn, vn)]
        rows = [[x * sc for x in base] for _, _, sc in steps]
        outs = [torch.empty_like(base[0]) for _ in steps]
        for j, (toks, ind, _) in enumerate(steps):
            eng.step(toks, ind, np.asarray(spec.req_new, np.int32), *rows[j], outs[j], groups="auto",
                     evict_tokens=T, overlap=True)
            if serial:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert eng.device_status() == 0
        eng.tree.check()
        results.append([to_host_f32(o) for o in outs])
    for j in range(len(steps)):
        assert np.array_equal(results[0][j], results[1][j]), f"step {j}"
    got = results[1][0]
    for b in range(w.batch):
        want, _ = oracle_rows(w, b)
        lo, hi = int(sum(spec.req_new[:b])), int(sum(spec.req_new[:b + 1]))
        compare(got[lo:hi], want, f"request {b}")


def test_host_buffer_decode_chunks_match_oracle():
    from prefix_cached_kv_radix_gb300.engine import _dev_from_host
    spec = small_decode(seed=27)
    w = W.generate(spec)
    prompts = [w.request_tokens(b) for b in range(w.batch)]
    ind = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
    toks = np.concatenate(prompts).astype(np.int32)
    q, kn, vn = w.stacked_new()
    eng = _engine_for(w)
    qd, kd, vd = (_dev_from_host(x, spec.dtype, eng.device) for x in (q, kn, vn))
    hq_, hk_, hv_ = (x.cpu().pin_memory() for x in (qd, kd, vd))
    out = torch.empty_like(qd)
    lse = torch.empty(qd.shape[0], spec.hq, dtype=torch.float32, device=eng.device)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    eng.step(toks, ind, spec.req_new, qd, kd, vd, out, lse, decode=True, host=(hq_, hk_, hv_, out_h, lse_h), chunks=4)
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    got, got_lse = out_h.float().numpy(), lse_h.numpy()
    for b in range(w.batch):
        want, wl = oracle_rows(w, b)
        compare(got[b:b + 1], want, f"request {b}")
        assert np.abs(got_lse[b:b + 1] - wl).max() <= TOL_LSE


@pytest.mark.gpu
def test_extend_persistent_grid_on_two_streams():
    """The extend kernel's persistent grid takes its items in order from a work counter per
    stream: the same extend call launched on two streams at once (more items than SMs, so the
    counters are used) gives, on each stream and on a third call after them, the output of the
    first call bit for bit, and that output matches the oracle."""
    spec = W.Spec("persist-2streams", "bf16", 32, 8, 128, 1 << 16, W.QWEN_VOCAB, 45,
                  seg_parent=[-1], seg_len=[300], histories=[0],
                  req_seg=[0] * 24, req_cached=[300] * 24, req_new=[128] * 24)
    w = W.generate(spec)
    eng, plan, dev, out, lse, _ = run_step(w)
    want = to_host_f32(out)
    q, _, _ = w.stacked_new()
    from prefix_cached_kv_radix_gb300.engine import _dev_from_host
    qd = _dev_from_host(q, spec.dtype, eng.device)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(out) for _ in streams]
    torch.cuda.synchronize()
    for _ in range(3):
        for st, o in zip(streams, outs):
            eng.extend(plan, dev, qd, o, stream=st.cuda_stream)
    torch.cuda.synchronize()
    again = torch.empty_like(out)
    eng.extend(plan, dev, qd, again)
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    for o in outs + [again]:
        assert np.array_equal(to_host_f32(o), want)
    for b in (0, 11, 23):
        lo, hi = b * 128, (b + 1) * 128
        o_want, _ = oracle_rows(w, b, rows=[0, 63, 127])
        compare(want[lo:hi][[0, 63, 127]], o_want, f"request {b}")
