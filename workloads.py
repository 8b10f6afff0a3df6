"""Seeded synthetic workloads for prefix-cached attention.

This module only draws random inputs and lays them out: token ids, per-segment
keys/values of the cached prefixes, and per-request queries/keys/values of the new
tokens.  It holds none of the method's arithmetic (no matching, no slot tables, no
attention), so both the CPU oracle and the CUDA path can consume what it produces.

A workload is a tree of cached *segments* (runs of tokens that earlier requests left
in the cache), a list of *histories* (segment paths inserted into the cache before the
measured step, in order) and a batch of *requests*.  A request follows the root path
of one segment for ``cached_len`` tokens and then appends ``n_new`` new tokens.

Shapes follow the five workloads of the prefix-caching pages:
  c1  tiny fp32 correctness case (64-token prefix, 4 x 8 new tokens, 4 heads x 64)
  c2  GPT-2 shaped shared system prompt (409 tokens, 64 x 7-8 new, 12 heads x 64)
  c3  few-shot branching tree (2048 root, 16 x 512 children, 8 x 128 new per child, GQA 32/8 x 128)
  c4  batched decode (256 requests, 1 token, contexts 1024..8192, 70% share 4096, GQA 32/8 x 128)
  c5  long multi-turn chat (32 branches of 32768, 90% hit, 1024 new, GQA 64/8 x 128)

Values: token ids uniform over the vocabulary; Q/K/V standard normal, rounded to
bf16 with round-to-nearest-even for bf16 workloads (kept as uint16 bit patterns),
plain float32 for fp32 workloads.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

GPT2_VOCAB = 50257
QWEN_VOCAB = 151936


# --------------------------------------------------------------------------- rounding
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); return uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- spec
@dataclass
class Spec:
    name: str
    dtype: str                    # "f32" or "bf16"
    hq: int
    hkv: int
    d: int
    num_slots: int
    vocab: int
    seed: int
    seg_parent: list              # parent segment id or -1
    seg_len: list                 # tokens per segment
    histories: list               # segment ids whose root paths are cached before the step
    req_seg: list                 # segment whose root path the request follows
    req_cached: list              # tokens of that path the request shares (a prefix of it)
    req_new: list                 # new tokens per request
    decode: bool = False          # one new token per request, attention by the decode kernel
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass
class Workload:
    spec: Spec
    seg_tokens: list = field(default_factory=list)   # int32 arrays
    seg_k: list = field(default_factory=list)        # [len, hkv, d] uint16 (bf16) or float32
    seg_v: list = field(default_factory=list)
    req_tokens: list = field(default_factory=list)   # new token ids per request (int32)
    req_q: list = field(default_factory=list)        # [n, hq, d]
    req_k: list = field(default_factory=list)        # [n, hkv, d]
    req_v: list = field(default_factory=list)

    # ---- layout helpers (concatenation only)
    def seg_path(self, s: int) -> list:
        path = []
        while s >= 0:
            path.append(s)
            s = self.spec.seg_parent[s]
        return path[::-1]

    def path_tokens(self, s: int) -> np.ndarray:
        return np.concatenate([self.seg_tokens[i] for i in self.seg_path(s)]).astype(np.int32)

    def path_kv(self, s: int):
        p = self.seg_path(s)
        return (np.concatenate([self.seg_k[i] for i in p]), np.concatenate([self.seg_v[i] for i in p]))

    @property
    def batch(self) -> int:
        return len(self.spec.req_seg)

    def request_prefix_tokens(self, b: int) -> np.ndarray:
        return self.path_tokens(self.spec.req_seg[b])[: self.spec.req_cached[b]]

    def request_tokens(self, b: int) -> np.ndarray:
        return np.concatenate([self.request_prefix_tokens(b), self.req_tokens[b]]).astype(np.int32)

    def request_kv(self, b: int):
        """Keys/values of request b's whole context in logical token order."""
        k, v = self.path_kv(self.spec.req_seg[b])
        c = self.spec.req_cached[b]
        return (np.concatenate([k[:c], self.req_k[b]]), np.concatenate([v[:c], self.req_v[b]]))

    def history_tokens(self, i: int) -> np.ndarray:
        return self.path_tokens(self.spec.histories[i])

    def history_kv(self, i: int):
        return self.path_kv(self.spec.histories[i])

    def qo_indptr(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.spec.req_new)]).astype(np.int64)

    def total_new(self) -> int:
        return int(sum(self.spec.req_new))

    def stacked_new(self):
        """Concatenate the new tokens' q, k, v over the batch: [T, h, d]."""
        return (np.concatenate(self.req_q), np.concatenate(self.req_k), np.concatenate(self.req_v))


# --------------------------------------------------------------------------- drawing
def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, *stream])


def _normal(seed: int, stream: tuple, shape, dtype: str):
    x = _rng(seed, *stream).standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(x).reshape(shape) if dtype == "bf16" else x


def _draw_first_distinct(rng, vocab: int, n: int, forbidden: set) -> np.ndarray:
    """n token ids; the first one avoids ``forbidden``; all n distinct when n <= vocab."""
    out = np.empty(n, dtype=np.int32)
    if n == 0:
        return out
    while True:
        t = int(rng.integers(0, vocab))
        if t not in forbidden:
            out[0] = t
            break
    if n > 1:
        out[1:] = rng.integers(0, vocab, size=n - 1)
    return out


def generate(spec: Spec, threads: int = 16) -> Workload:
    """Draw every token id and tensor of ``spec`` from its seed (deterministic)."""
    w = Workload(spec)
    nseg = len(spec.seg_parent)
    tok_rng = _rng(spec.seed, 0)
    # Segment tokens: siblings (and root segments) start with distinct tokens, so the
    # cached tree branches exactly at segment ends.
    first_of_children: dict = {}
    for s in range(nseg):
        par = spec.seg_parent[s]
        used = first_of_children.setdefault(par, set())
        toks = _draw_first_distinct(tok_rng, spec.vocab, spec.seg_len[s], used)
        if len(toks):
            used.add(int(toks[0]))
        w.seg_tokens.append(toks)
    # Request tokens: the first new token differs from the cached continuation at the
    # divergence point and from every sibling request diverging at the same point.
    lens_path = {}
    for b in range(len(spec.req_seg)):
        s, c = spec.req_seg[b], spec.req_cached[b]
        if s not in lens_path:
            lens_path[s] = w.path_tokens(s) if s >= 0 else np.zeros(0, np.int32)
        path = lens_path[s]
        key = (s, c)
        forb = first_of_children.setdefault(("req", key), set())
        if c < len(path):
            forb.add(int(path[c]))
        # At the end of a segment on the path (or at the very start): avoid every child
        # segment's first token there.
        if c == 0:
            forb |= first_of_children.get(-1, set())
        end = 0
        for seg in (w.seg_path(s) if s >= 0 else []):
            end += spec.seg_len[seg]
            if end == c:
                forb |= first_of_children.get(seg, set())
        n = spec.req_new[b]
        if n <= spec.vocab // 4:
            toks = np.empty(n, np.int32)
            if n:
                while True:
                    cand = tok_rng.choice(spec.vocab, size=n, replace=False).astype(np.int32)
                    if int(cand[0]) not in forb:
                        toks = cand
                        break
        else:
            toks = _draw_first_distinct(tok_rng, spec.vocab, n, forb)
        if n:
            forb.add(int(toks[0]))
        w.req_tokens.append(toks)

    # Tensors, one independent stream per segment / request so they can be drawn in parallel.
    def seg_job(s):
        shp = (spec.seg_len[s], spec.hkv, spec.d)
        return _normal(spec.seed, (1, s, 0), shp, spec.dtype), _normal(spec.seed, (1, s, 1), shp, spec.dtype)

    def req_job(b):
        n = spec.req_new[b]
        return (_normal(spec.seed, (2, b, 0), (n, spec.hq, spec.d), spec.dtype),
                _normal(spec.seed, (2, b, 1), (n, spec.hkv, spec.d), spec.dtype),
                _normal(spec.seed, (2, b, 2), (n, spec.hkv, spec.d), spec.dtype))

    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        for k, v in ex.map(seg_job, range(nseg)):
            w.seg_k.append(k)
            w.seg_v.append(v)
        for q, k, v in ex.map(req_job, range(len(spec.req_seg))):
            w.req_q.append(q)
            w.req_k.append(k)
            w.req_v.append(v)
    return w


# --------------------------------------------------------------------------- specs
def spec_shared_prompt(name, dtype, hq, hkv, d, num_slots, vocab, seed, prefix, new_lens, note=""):
    """One cached prefix shared by every request (c1, c2 and small variants)."""
    b = len(new_lens)
    return Spec(name, dtype, hq, hkv, d, num_slots, vocab, seed,
                seg_parent=[-1], seg_len=[prefix], histories=[0],
                req_seg=[0] * b, req_cached=[prefix] * b, req_new=list(new_lens), note=note)


def spec_branching(name, dtype, hq, hkv, d, num_slots, vocab, seed, root, n_children, child_len,
                   leaves_per_child, n_new, note=""):
    """Root prefix, children under it, leaf requests per child (c3 and small variants)."""
    parent = [-1] + [0] * n_children
    seg_len = [root] + [child_len] * n_children
    req_seg, req_cached, req_new = [], [], []
    for c in range(n_children):
        for _ in range(leaves_per_child):
            req_seg.append(1 + c)
            req_cached.append(root + child_len)
            req_new.append(n_new)
    return Spec(name, dtype, hq, hkv, d, num_slots, vocab, seed, parent, seg_len,
                histories=list(range(1, n_children + 1)), req_seg=req_seg, req_cached=req_cached,
                req_new=req_new, note=note)


def spec_decode(name, dtype, hq, hkv, d, num_slots, vocab, seed, batch, share_frac, shared_len,
                min_len, max_len, note=""):
    """Batched decode: a fraction of requests share one cached prefix (c4 and small variants).

    Sharers are chosen by a seeded permutation; they draw L ~ U[shared_len+1, max_len],
    the others L ~ U[min_len, max_len].  L counts the decode token, so the cached context is
    L-1 tokens and one new token is appended.
    """
    rng = _rng(seed, 3)
    n_share = int(round(share_frac * batch))
    perm = rng.permutation(batch)
    sharer = np.zeros(batch, bool)
    sharer[perm[:n_share]] = True
    own = rng.integers(min_len, max_len + 1, size=batch)
    shr = rng.integers(shared_len + 1, max_len + 1, size=batch) if n_share else own
    lens = np.where(sharer, shr, own)
    parent, seg_len = [], []
    if n_share:
        parent.append(-1)
        seg_len.append(shared_len)
    req_seg, req_cached = [], []
    for b in range(batch):
        L = int(lens[b])
        if sharer[b]:
            priv = L - 1 - shared_len
            if priv > 0:
                parent.append(0)
                seg_len.append(priv)
                req_seg.append(len(seg_len) - 1)
            else:
                req_seg.append(0)
        else:
            parent.append(-1)
            seg_len.append(L - 1)
            req_seg.append(len(seg_len) - 1)
        req_cached.append(L - 1)
    parents = set(parent)
    hist = [s for s in range(len(seg_len)) if s not in parents]   # leaf segments
    return Spec(name, dtype, hq, hkv, d, num_slots, vocab, seed, parent, seg_len,
                histories=hist, req_seg=req_seg, req_cached=req_cached, req_new=[1] * batch,
                decode=True, note=note)


def spec_multiturn(name, dtype, hq, hkv, d, num_slots, vocab, seed, branches, branch_len, hit_len,
                   n_new, note=""):
    """Independent conversation branches; each request follows its branch for hit_len tokens
    and then diverges with n_new new tokens (c5 and small variants)."""
    return Spec(name, dtype, hq, hkv, d, num_slots, vocab, seed,
                seg_parent=[-1] * branches, seg_len=[branch_len] * branches,
                histories=list(range(branches)), req_seg=list(range(branches)),
                req_cached=[hit_len] * branches, req_new=[n_new] * branches, note=note)


def config(name: str) -> Spec:
    """The five named workloads."""
    if name == "c1":
        return spec_shared_prompt("c1", "f32", 4, 4, 64, 512, GPT2_VOCAB, 1, 64, [8] * 4,
                                  note="tiny fp32 correctness case")
    if name == "c2":
        rng = _rng(2, 4)
        lens = rng.integers(7, 9, size=64).tolist()
        return spec_shared_prompt("c2", "bf16", 12, 12, 64, 65536, GPT2_VOCAB, 2, 409, lens,
                                  note="GPT-2 shaped shared system prompt")
    if name == "c3":
        return spec_branching("c3", "bf16", 32, 8, 128, 1 << 20, QWEN_VOCAB, 3, 2048, 16, 512, 8, 128,
                              note="few-shot branching tree")
    if name == "c4":
        return spec_decode("c4", "bf16", 32, 8, 128, 1 << 21, QWEN_VOCAB, 4, 256, 0.7, 4096, 1024, 8192,
                           note="batched decode")
    if name == "c5":
        return spec_multiturn("c5", "bf16", 64, 8, 128, 1 << 22, QWEN_VOCAB, 5, 32, 32768,
                              int(0.9 * 32768), 1024, note="long multi-turn chat")
    raise KeyError(name)


CONFIG_NAMES = ("c1", "c2", "c3", "c4", "c5")


def take_requests(spec: Spec, n: int) -> Spec:
    """The first n requests of ``spec`` with the segments on their paths (renumbered, parents
    kept) and only those histories: the same per-request shapes at a smaller footprint, for
    profiling captures.  Token and tensor values differ from the full workload's (they are
    drawn per segment and request index)."""
    n = max(0, min(n, len(spec.req_seg)))
    keep = set()
    for sg in spec.req_seg[:n]:
        while sg >= 0 and sg not in keep:
            keep.add(sg)
            sg = spec.seg_parent[sg]
    order = sorted(keep)
    new_id = {old: i for i, old in enumerate(order)}
    remap = lambda sg: new_id[sg] if sg >= 0 else -1
    return Spec(f"{spec.name}-first{n}", spec.dtype, spec.hq, spec.hkv, spec.d, spec.num_slots, spec.vocab, spec.seed,
                seg_parent=[remap(spec.seg_parent[o]) for o in order], seg_len=[spec.seg_len[o] for o in order],
                histories=[new_id[h] for h in spec.histories if h in keep],
                req_seg=[remap(x) for x in spec.req_seg[:n]], req_cached=list(spec.req_cached[:n]),
                req_new=list(spec.req_new[:n]), decode=spec.decode,
                note=f"{spec.note}, first {n} requests")


# ---------------------------------------------------------------------------- request traces
@dataclass
class Session:
    """One conversation: a shared prefix (system prompt or few-shot block, by id), then turns
    of (user tokens, reply tokens).  Turn t's request is prefix + every earlier turn's user and
    reply tokens + turn t's user tokens; its reply is generated after it."""
    prefix_id: int
    start: int                       # arrival step of the first turn
    turns: list = field(default_factory=list)


@dataclass
class Trace:
    prefixes: list                   # token arrays, by prefix id
    sessions: list                   # Session

    def request(self, s: int, t: int) -> np.ndarray:
        ses = self.sessions[s]
        parts = [self.prefixes[ses.prefix_id]]
        for u, r in ses.turns[:t]:
            parts += [u, r]
        parts.append(ses.turns[t][0])
        return np.concatenate(parts).astype(np.int32)

    def sequence(self, s: int, t: int) -> np.ndarray:
        """The request followed by its reply: what the cache holds once the turn is done."""
        return np.concatenate([self.request(s, t), self.sessions[s].turns[t][1]]).astype(np.int32)


def chat_trace(seed: int, vocab: int = 151936, n_system: int = 4, n_fewshot: int = 3, n_chats: int = 48,
               n_questions: int = 96, horizon: int = 64, scale: int = 1) -> Trace:
    """Seeded request trace in the shape of the "SGLang" page's walk-through: chat sessions that
    share a few system prompts and grow turn by turn (each turn's prompt holds the whole
    conversation so far), and few-shot question sets that share a long examples block.  Token
    ids are uniform; lengths are uniform in the ranges below; arrivals are uniform over
    `horizon` steps; `scale` divides every length (small traces for exhaustive checks)."""
    rng = _rng(seed, 31)

    def n(lo, hi):
        return int(rng.integers(max(lo // scale, 1), max(hi // scale, 1) + 1))

    prefixes = [rng.integers(0, vocab, size=n(256, 1024)).astype(np.int32) for _ in range(n_system)]
    prefixes += [rng.integers(0, vocab, size=n(512, 2048)).astype(np.int32) for _ in range(n_fewshot)]
    sessions = []
    for _ in range(n_chats):
        s = Session(int(rng.integers(0, n_system)), int(rng.integers(0, horizon)))
        for _t in range(int(rng.integers(2, 7))):
            s.turns.append((rng.integers(0, vocab, size=n(16, 128)).astype(np.int32),
                            rng.integers(0, vocab, size=n(32, 256)).astype(np.int32)))
        sessions.append(s)
    for _ in range(n_questions):
        s = Session(n_system + int(rng.integers(0, n_fewshot)), int(rng.integers(0, horizon)))
        s.turns.append((rng.integers(0, vocab, size=n(16, 64)).astype(np.int32),
                        rng.integers(0, vocab, size=n(8, 32)).astype(np.int32)))
        sessions.append(s)
    return Trace(prefixes, sessions)
