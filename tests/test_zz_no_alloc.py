"""decode_attention_noalloc: the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory per call (a plug-in whose host
application already owns the GPU's memory, a serving loop that must not stall on
cudaMalloc/cudaFree, a plain C caller without an allocator for the workspace).  Its
scratch is one static device array shared by every call.  It runs the same kernels as
decode_attention on the same inputs, so its output and lse must equal the workspace
call's bit for bit, and the oracle's within the attention tolerance.  This file is
collected last on purpose: if it fails, a run that stops at the first failure has already
run every other test.  It builds everything it needs itself, so it also passes alone in a
fresh process.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_cases import TOL_LSE, compare, oracle_rows, run_step, to_host_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_cached_kv_radix_gb300 import api
    api.load()


def _check_against_oracle(w, out, lse):
    got, got_lse = to_host_f32(out), lse.cpu().numpy()
    for b in range(w.batch):
        want, wl = oracle_rows(w, b)
        compare(got[b:b + 1], want, f"request {b}")
        assert np.abs(got_lse[b:b + 1] - wl).max() <= TOL_LSE, f"request {b}: lse"


@pytest.mark.parametrize("use_groups", [False, True])
def test_noalloc_decode_equals_workspace_decode_twice(use_groups):
    from prefix_cached_kv_radix_gb300 import api
    spec = W.spec_decode("noalloc", "bf16", 32, 8, 128, 1 << 16, W.QWEN_VOCAB, 31, batch=20, share_frac=0.6,
                         shared_len=500, min_len=1, max_len=2500)
    w = W.generate(spec)
    eng, plan, dev, ref_out, ref_lse, grp = run_step(w, groups=use_groups)
    assert eng.device_status() == 0
    assert (grp is not None) == use_groups
    need = api.decode_workspace_bytes(eng.desc, plan.batch, plan.max_kv_len, grp)
    assert 0 < need <= api.RX_DECODE_NOALLOC_SCRATCH_BYTES
    q = torch.empty(plan.batch, spec.hq, spec.d, dtype=torch.bfloat16, device="cuda")
    q.copy_(torch.from_numpy(np.concatenate(w.req_q).view(np.int16)).view(torch.bfloat16))
    ref_o = ref_out.view(torch.int16).cpu().numpy()
    ref_l = ref_lse.cpu().numpy()
    _check_against_oracle(w, ref_out, ref_lse)
    for call in range(2):                       # two calls in a row share the static scratch
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        # the second call passes the slot table as a raw device address with its stride
        r2t = dev["r2t"] if call == 0 else dev["r2t"].data_ptr()
        api.decode_attention_noalloc(eng.desc, plan.batch, q, r2t, dev["kv_lens"], eng.k_pool, eng.v_pool,
                                     out, lse, plan.max_kv_len, eng.status, groups=grp,
                                     r2t_stride=None if call == 0 else dev["r2t"].shape[1])
        torch.cuda.synchronize()
        assert eng.device_status() == 0
        assert np.array_equal(out.view(torch.int16).cpu().numpy(), ref_o), f"call {call}: output differs"
        assert np.array_equal(lse.cpu().numpy(), ref_l), f"call {call}: lse differs"
        _check_against_oracle(w, out, lse)


def test_noalloc_fp32_needs_no_scratch_at_any_batch():
    """The fp32 path runs on CUDA cores without a workspace: decode_workspace_bytes is 0, so a
    batch far beyond what the split-KV scratch could hold is accepted, and its results equal
    the workspace-free decode_attention call's bit for bit."""
    from prefix_cached_kv_radix_gb300 import api
    spec = W.spec_decode("noalloc-f32", "f32", 8, 2, 64, 1 << 15, W.QWEN_VOCAB, 32, batch=600, share_frac=0.5,
                         shared_len=24, min_len=1, max_len=40)
    w = W.generate(spec)
    eng, plan, dev, ref_out, ref_lse, _ = run_step(w)
    assert eng.device_status() == 0
    big = 1 << 16
    assert api.decode_workspace_bytes(eng.desc, plan.batch, big) == 0
    bf = api.make_desc(api.RX_BF16, 32, 8, 128, 1 << 20, 128 ** -0.5)
    assert api.decode_workspace_bytes(bf, plan.batch, big) > api.RX_DECODE_NOALLOC_SCRATCH_BYTES
    q = torch.from_numpy(np.concatenate(w.req_q)).cuda()
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        api.decode_attention_noalloc(eng.desc, plan.batch, q, dev["r2t"], dev["kv_lens"], eng.k_pool, eng.v_pool,
                                     out, lse, big, eng.status)
        torch.cuda.synchronize()
        assert eng.device_status() == 0
        assert np.array_equal(out.cpu().numpy(), ref_out.cpu().numpy()), f"call {call}"
        assert np.array_equal(lse.cpu().numpy(), ref_lse.cpu().numpy()), f"call {call}"
    for b in (0, 1, plan.batch // 2, plan.batch - 1):
        want, wl = oracle_rows(w, b)
        compare(to_host_f32(out)[b:b + 1], want, f"fp32 request {b}")
        assert np.abs(lse.cpu().numpy()[b:b + 1] - wl).max() <= TOL_LSE


def test_noalloc_rejects_a_batch_beyond_the_static_scratch():
    from prefix_cached_kv_radix_gb300 import api
    desc = api.make_desc(api.RX_BF16, 32, 8, 128, 1 << 20, 128 ** -0.5)
    batch, max_len = 512, 32768
    assert api.decode_workspace_bytes(desc, batch, max_len) > api.RX_DECODE_NOALLOC_SCRATCH_BYTES
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = torch.zeros(batch, 32, 128, dtype=torch.bfloat16, device="cuda")
    r2t = torch.zeros(batch, 8, dtype=torch.int32, device="cuda")
    lens = torch.ones(batch, dtype=torch.int32, device="cuda")
    pool = torch.zeros(16, 8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.RxError) as e:
        api.decode_attention_noalloc(desc, batch, q, r2t, lens, pool, pool, torch.empty_like(q), None, max_len, t)
    assert e.value.code == api.RX_EINVAL and "static scratch" in str(e.value)
