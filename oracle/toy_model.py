"""Toy causal language model for the cached-versus-recomputed check (test infrastructure only).

"Prompt Caching" (Ultralytics glossary), "How prompt caching works": the page's GPT-2
example prefills a 409-token system prompt once, then runs each question's tokens alone
on top of the cached keys/values, and checks that the last position's next-token scores
equal a full recomputation of the whole prompt (allclose, atol 1e-3); it prints
"Computed 8 of 417 tokens" and "Computed 7 of 416 tokens".  No trained weights are
available here, so this model has random weights of a small GPT-like shape (token and
position embeddings, pre-norm blocks of causal multi-head attention and an MLP, tied
output head).  Attention goes through the oracle's plain causal attention.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_rows


def _layernorm(x):
    mu = x.mean(-1, keepdims=True)
    var = ((x - mu) ** 2).mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(var + 1e-5)


def _gelu(x):
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


class ToyCausalLM:
    def __init__(self, seed: int, vocab: int = 50257, d_model: int = 64, n_heads: int = 4,
                 n_layers: int = 2, max_pos: int = 1024):
        rng = np.random.default_rng([seed, 77])
        self.h, self.dh = n_heads, d_model // n_heads
        self.wte = rng.normal(0.0, 0.02, (vocab, d_model))
        self.wpe = rng.normal(0.0, 0.01, (max_pos, d_model))
        s = 1.0 / np.sqrt(d_model)
        self.layers = [dict(wq=rng.normal(0, s, (d_model, d_model)), wk=rng.normal(0, s, (d_model, d_model)),
                            wv=rng.normal(0, s, (d_model, d_model)), wo=rng.normal(0, s, (d_model, d_model)),
                            w1=rng.normal(0, s, (d_model, 4 * d_model)),
                            w2=rng.normal(0, s / 2, (4 * d_model, d_model)))
                       for _ in range(n_layers)]

    def forward(self, ids, past=None):
        """Run ``ids`` on top of the per-layer cache ``past`` (list of (K, V)) or from scratch.

        Returns (logits [n, vocab], present) where present holds each layer's keys/values
        for every position processed so far, in logical order."""
        ids = np.asarray(ids)
        n = len(ids)
        start = 0 if past is None else past[0][0].shape[0]
        x = self.wte[ids] + self.wpe[start:start + n]
        present = []
        pos = np.arange(start, start + n, dtype=np.int64)
        for li, L in enumerate(self.layers):
            hdn = _layernorm(x)
            q = (hdn @ L["wq"]).reshape(n, self.h, self.dh)
            k = (hdn @ L["wk"]).reshape(n, self.h, self.dh)
            v = (hdn @ L["wv"]).reshape(n, self.h, self.dh)
            if past is not None:
                k = np.concatenate([past[li][0], k])
                v = np.concatenate([past[li][1], v])
            present.append((k, v))
            o, _ = attention_rows(q.astype(np.float32), pos, k.astype(np.float32), v.astype(np.float32),
                                  1.0 / np.sqrt(self.dh))
            x = x + o.reshape(n, -1).astype(np.float64) @ L["wo"]
            x = x + _gelu(_layernorm(x) @ L["w1"]) @ L["w2"]
        return _layernorm(x) @ self.wte.T, present
