"""Combining softmax attention over disjoint key sets (test infrastructure only).

Not on the pages: the pages define only the full causal attention.  A split of the keys
into disjoint parts is exact because softmax attention over a union can be rebuilt from
each part's normalised output o_s and log-sum-exp lse_s:
    M = max_s lse_s,  w_s = exp(lse_s - M),
    o = sum_s w_s o_s / sum_s w_s,   lse = M + log(sum_s w_s).
Written out in fp64 from that definition.
"""
from __future__ import annotations

import numpy as np


def merge_states(outs, lses):
    """outs: [S, ..., d] partial outputs; lses: [S, ...] their log-sum-exp values."""
    outs = np.asarray(outs, np.float64)
    lses = np.asarray(lses, np.float64)
    M = lses.max(axis=0)
    w = np.exp(lses - M)
    den = w.sum(axis=0)
    o = (w[..., None] * outs).sum(axis=0) / den[..., None]
    return o, M + np.log(den)
