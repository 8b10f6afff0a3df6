"""Helpers for the GPU parity tests: run a workload through the library and compute what
the oracle says it must produce (expected slots from the list matcher and the replayed
allocator; expected attention from the fp64 oracle over logical-order K/V)."""
import numpy as np
import torch

import oracle
import workloads as W

TOL_MAX_ABS = 2e-2     # attention outputs, bf16 in / fp32 accumulate
TOL_MEAN_ABS = 2e-3
TOL_REL_FRO = 1e-2     # per (request, head): ||got - want|| / ||want||
TOL_LSE = 1e-3


def f32(a, dtype):
    return W.bf16_bits_to_f32(a) if dtype == "bf16" else np.asarray(a, np.float32)


def to_host_f32(t):
    return t.float().cpu().numpy()


def expected_slots(w):
    """Oracle replay of populate + plan: (prefix slot lists, new slot lists, P per request)."""
    s = w.spec
    alloc = oracle.SlotAllocator(s.num_slots, s.seed)
    lm = oracle.ListMatcher()
    for i in range(len(s.histories)):
        toks = w.history_tokens(i)
        m, sl = lm.match(toks)
        new = alloc.alloc(len(toks) - m)
        lm.add(toks, np.concatenate([sl, new]))
    pre, P = [], []
    for b in range(w.batch):
        m, sl = lm.match(w.request_tokens(b))
        pre.append(sl)
        P.append(m)
    T = w.total_new()
    new = alloc.alloc(T)
    qo = w.qo_indptr()
    return pre, [new[qo[b]:qo[b + 1]] for b in range(w.batch)], np.array(P)


def run_step(w, engine=None, groups=False, lse=True, poison=True):
    """Populate the cache with the workload's histories, then run one step on the GPU."""
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine, _dev_from_host
    s = w.spec
    eng = engine or PrefixCacheEngine(s.dtype, s.hq, s.hkv, s.d, s.num_slots, s.seed, poison=poison)
    for i in range(len(s.histories)):
        k, v = w.history_kv(i)
        eng.populate(w.history_tokens(i), k, v)
    plan = eng.plan([w.request_tokens(b) for b in range(w.batch)], s.req_new, groups=groups)
    dev = eng.upload(plan)
    q, kn, vn = w.stacked_new()
    qd, kd, vd = (_dev_from_host(x, s.dtype, eng.device) for x in (q, kn, vn))
    out = torch.empty_like(qd)
    lse_t = torch.empty(qd.shape[0], s.hq, dtype=torch.float32, device=eng.device) if lse else None
    eng.write(plan, dev, kd, vd)
    grp = None
    if s.decode:
        grp = eng.groups(plan, dev) if groups else None
        eng.decode(plan, dev, qd, out, lse_t, groups=grp)
    else:
        grp = eng.groups(plan, dev)
        eng.extend(plan, dev, qd, out, lse_t)
    torch.cuda.synchronize()
    return eng, plan, dev, out, lse_t, grp


def oracle_rows(w, b, rows=None, threads=0):
    """Oracle attention for request b's new rows (all, or the given row indices)."""
    s = w.spec
    k, v = w.request_kv(b)
    k, v = f32(k, s.dtype), f32(v, s.dtype)
    q = f32(w.req_q[b], s.dtype)
    P = s.req_cached[b]
    idx = np.arange(s.req_new[b]) if rows is None else np.asarray(rows)
    o, l = oracle.attention_rows(q[idx], P + idx, k, v, s.scale, threads)
    return o, l


def compare(got, want, what="", max_abs=TOL_MAX_ABS):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= TOL_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    # relative Frobenius per head (last axis = head_dim, second to last = head)
    num = np.sqrt((err ** 2).sum(axis=(0, -1)))
    den = np.sqrt((want ** 2).sum(axis=(0, -1)))
    rel = num / np.maximum(den, 1e-30)
    assert rel.max() <= TOL_REL_FRO, f"{what}: relative Frobenius err {rel.max():.3e}"
    return err.max(), err.mean(), rel.max()
