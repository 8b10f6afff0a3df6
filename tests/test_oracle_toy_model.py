"""The claim prefix caching rests on, reproduced on the oracle with a random-weight model.

"Prompt Caching" (Ultralytics glossary), "How prompt caching works": prefilling a
409-token prompt once and running only a question's tokens on top of the cached
keys/values gives the same next-token scores as recomputing the whole prompt (the page
prints "Computed 8 of 417 tokens ... True" and "Computed 7 of 416 tokens ... True",
compared with allclose at atol 1e-3).  Trained GPT-2 weights are not available, so a
seeded toy causal model stands in; the counts and tolerance come from the golden file.
"""
import copy
import json
import os

import numpy as np

from oracle.toy_model import ToyCausalLM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prompt_caching_gpt2_counts.json")


def test_cached_prefix_gives_full_recompute_scores():
    g = json.load(open(GOLDEN))
    model = ToyCausalLM(seed=409)
    rng = np.random.default_rng(2024)
    prefix = rng.integers(0, 50257, size=g["prefix_tokens"])
    _, cache = model.forward(prefix)
    for case in g["cases"]:
        q = rng.integers(0, 50257, size=case["computed"])
        cached, _ = model.forward(q, past=copy.deepcopy(cache))
        full, _ = model.forward(np.concatenate([prefix, q]))
        same = bool(np.allclose(cached[-1], full[-1], atol=g["atol"]))
        assert same == case["same_next_token_scores"]
        assert len(q) + len(prefix) == case["total"]
        assert len(q) / case["total"] < g["fraction_computed_below"]
        # in practice the two agree to rounding, far inside the page's tolerance
        assert np.abs(cached[-1] - full[-1]).max() < 1e-5
        # every new row, not just the last, matches the full computation
        np.testing.assert_allclose(cached, full[len(prefix):], atol=1e-5, rtol=0)


def test_a_wrong_cache_is_detected():
    # The comparison has teeth: a cache of a different prefix changes the scores.
    model = ToyCausalLM(seed=409)
    rng = np.random.default_rng(7)
    prefix = rng.integers(0, 50257, size=64)
    other = prefix.copy()
    other[10] = (other[10] + 1) % 50257
    _, wrong_cache = model.forward(other)
    q = rng.integers(0, 50257, size=8)
    cached, _ = model.forward(q, past=wrong_cache)
    full, _ = model.forward(np.concatenate([prefix, q]))
    assert np.abs(cached[-1] - full[-1]).max() > 1e-5
