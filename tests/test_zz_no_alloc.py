"""decode_attention_noalloc: the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory per call (a plug-in whose host
application already owns the GPU's memory, a serving loop that must not stall on
cudaMalloc/cudaFree, a plain C caller without an allocator for the workspace).  Its
scratch is one static device array shared by every call.  This file is collected last on
purpose: if it fails, a run that stops at the first failure has already run every other
test.  It builds everything it needs itself, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_cases import TOL_LSE, TOL_MAX_ABS, TOL_MEAN_ABS, run_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefix_cached_kv_radix_gb300 import api
    api.load()


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
    qs = np.concatenate(w.req_q)
    q.copy_(torch.from_numpy(qs.view(np.int16)).view(torch.bfloat16))
    ref = ref_out.float()
    for call in range(2):                       # two calls in a row share the static scratch
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        api.decode_attention_noalloc(eng.desc, plan.batch, q, dev["r2t"], dev["kv_lens"], eng.k_pool, eng.v_pool,
                                     out, lse, plan.max_kv_len, eng.status, groups=grp)
        torch.cuda.synchronize()
        assert eng.device_status() == 0
        err = (out.float() - ref).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= TOL_MAX_ABS and err.mean().item() <= TOL_MEAN_ABS, (call, err.max().item())
        assert (lse - ref_lse).abs().max().item() <= TOL_LSE


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
