"""The synthetic workload generator's request subset (used for smaller profiling captures)."""
import numpy as np

import workloads as W


def test_take_requests_keeps_shapes_and_paths():
    for name in ("c2", "c3", "c4", "c5"):
        full = W.config(name)
        sub = W.take_requests(full, 3)
        assert sub.req_cached == full.req_cached[:3] and sub.req_new == full.req_new[:3]
        assert (sub.hq, sub.hkv, sub.d, sub.dtype) == (full.hq, full.hkv, full.d, full.dtype)
        # every kept segment's parent is kept and numbered before it
        for i, par in enumerate(sub.seg_parent):
            assert par < i
        w = W.generate(sub)
        for b in range(3):
            path = w.path_tokens(sub.req_seg[b])
            assert len(path) >= sub.req_cached[b]             # the cached part lies on the path
            assert len(w.req_tokens[b]) == sub.req_new[b]
        # the histories cache every request's path
        w0 = W.Workload(sub)
        on_history = set()
        for h in sub.histories:
            on_history.update(w0.seg_path(h))
        for b in range(3):
            assert sub.req_cached[b] == 0 or sub.req_seg[b] in on_history
