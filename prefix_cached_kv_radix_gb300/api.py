"""Thin Python binding of libradixattn.so (ctypes).

Argument marshalling only: every step runs in the library (host C++ radix tree, CUDA
kernels).  Names follow the C ABI in include/radix_attn.h.  Device buffers are torch
tensors on the current CUDA device; the call is enqueued on the given stream (default:
torch's current stream).  A missing library raises at once: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libradixattn.so")

RX_OK, RX_EINVAL, RX_ENOMEM, RX_ECUDA, RX_ELOCKED, RX_ETIMEOUT, RX_EDEVICE = 0, -1, -2, -3, -4, -5, -6
RX_DEV_OK, RX_DEV_BAD_SLOT, RX_DEV_BAD_LENGTH, RX_DEV_TIMEOUT = 0, 1, 2, 3
RX_F32, RX_BF16 = 0, 1
RX_DECODE_NOALLOC_SCRATCH_BYTES = 32 << 20   # include/radix_attn.h

EXPORTS = ("radix_create", "radix_destroy", "match_prefix", "match_prefix_len", "match_prefix_len_batch", "radix_set_page_size",
           "radix_lock", "radix_unlock", "alloc_slots",
           "free_slots", "insert", "evict", "match_prefix_batch", "insert_batch", "insert_batch_at", "radix_lock_batch",
           "radix_unlock_batch", "radix_stats", "radix_check",
           "radix_shared_groups", "rx_step_stage_bytes", "rx_step_plan", "rx_step_finish",
           "rx_step_workspace_bytes", "rx_step_launch", "rx_step_prefetch", "rx_step_ranges", "rx_stage_wait", "rx_step_run",
           "kv_pool_write", "prefix_extend_attention", "extend_workspace_bytes", "decode_workspace_bytes",
           "decode_attention",
           "decode_attention_noalloc",
           "rx_last_error", "rx_version", "rx_wait_selftest", "rx_set_tracing")


class RxError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed ({code}): {msg}")
        self.code = code


class rx_attn_desc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("num_slots", ctypes.c_int64), ("scale", ctypes.c_float)]


class rx_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "match_calls", "match_query_tokens", "match_hit_tokens", "insert_calls", "inserted_tokens",
        "evicted_tokens", "node_count", "cached_tokens", "free_slots", "num_slots")]


class rx_shared_groups(ctypes.Structure):
    _fields_ = [("num_groups", ctypes.c_int32), ("max_group_size", ctypes.c_int32),
                ("d_group_indptr", ctypes.c_void_p), ("d_group_members", ctypes.c_void_p),
                ("d_group_len", ctypes.c_void_p), ("max_group_len", ctypes.c_int32),
                ("max_group_rows", ctypes.c_int32)]


class rx_step_layout(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_qo_len", ctypes.c_int32), ("max_kv_len", ctypes.c_int32),
                ("stride", ctypes.c_int32), ("total_new", ctypes.c_int64), ("total_prefix", ctypes.c_int64),
                ("bytes", ctypes.c_int64), ("off_prefix_slots", ctypes.c_int64), ("off_prefix_indptr", ctypes.c_int64),
                ("off_new_slots", ctypes.c_int64), ("off_qo_indptr", ctypes.c_int64),
                ("off_prefix_lens", ctypes.c_int64), ("off_kv_lens", ctypes.c_int64),
                ("num_groups", ctypes.c_int32), ("max_group_size", ctypes.c_int32),
                ("max_group_len", ctypes.c_int32), ("max_group_rows", ctypes.c_int32),
                ("off_grp_indptr", ctypes.c_int64), ("off_grp_members", ctypes.c_int64),
                ("off_grp_len", ctypes.c_int64)]


RX_GROUPS_NONE, RX_GROUPS_ALWAYS, RX_GROUPS_AUTO = 0, 1, 2


class rx_step_io(ctypes.Structure):
    _fields_ = [("d_q", ctypes.c_void_p), ("d_k_new", ctypes.c_void_p), ("d_v_new", ctypes.c_void_p),
                ("d_k_pool", ctypes.c_void_p), ("d_v_pool", ctypes.c_void_p), ("d_out", ctypes.c_void_p),
                ("d_lse", ctypes.c_void_p), ("d_stage", ctypes.c_void_p), ("d_stage_bytes", ctypes.c_size_t),
                ("d_r2t", ctypes.c_void_p), ("r2t_elems", ctypes.c_int64), ("d_workspace", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t), ("d_status", ctypes.c_void_p), ("decode", ctypes.c_int32),
                ("h_q", ctypes.c_void_p), ("h_k_new", ctypes.c_void_p), ("h_v_new", ctypes.c_void_p),
                ("h_out", ctypes.c_void_p), ("h_lse", ctypes.c_void_p), ("chunks", ctypes.c_int32),
                ("overlap", ctypes.c_int32)]


class rx_step_args(ctypes.Structure):
    _fields_ = [("tree", ctypes.c_void_p), ("desc", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("group_mode", ctypes.c_int32), ("tokens", ctypes.c_void_p), ("tok_indptr", ctypes.c_void_p),
                ("n_new", ctypes.c_void_p), ("heads_per_kv", ctypes.c_int32), ("pad0", ctypes.c_int32),
                ("min_shared", ctypes.c_int64), ("h_stage", ctypes.c_void_p), ("stage_cap", ctypes.c_size_t),
                ("io", ctypes.c_void_p), ("evict_tokens", ctypes.c_int64), ("out_last", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("out_evicted", ctypes.c_void_p), ("stream", ctypes.c_void_p)]


_lib = None
P = ctypes.c_void_p
I32, I64, U64, SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t


def load(path: str = LIB_PATH):
    """Load the library (build it first with prefix_cached_kv_radix_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libradixattn.so is not built ({path}); run "
                           "`python -m prefix_cached_kv_radix_gb300.build`")
    lib = ctypes.CDLL(path)
    sig = {
        "radix_create": (ctypes.c_int, [I64, U64, P]),
        "radix_destroy": (None, [P]),
        "match_prefix": (ctypes.c_int, [P, P, I64, P, P, P]),
        "match_prefix_len": (ctypes.c_int, [P, P, I64, P]),
        "match_prefix_len_batch": (ctypes.c_int, [P, I32, P, P, P]),
        "radix_set_page_size": (ctypes.c_int, [P, I64]),
        "radix_lock": (ctypes.c_int, [P, I64]),
        "radix_unlock": (ctypes.c_int, [P, I64]),
        "alloc_slots": (ctypes.c_int, [P, I64, P]),
        "free_slots": (ctypes.c_int, [P, P, I64]),
        "insert": (ctypes.c_int, [P, P, P, I64, P, P]),
        "evict": (ctypes.c_int, [P, I64, P, I64, P]),
        "match_prefix_batch": (ctypes.c_int, [P, I32, P, P, P, P, P]),
        "insert_batch": (ctypes.c_int, [P, I32, P, P, P, P, P]),
        "insert_batch_at": (ctypes.c_int, [P, I32, P, P, P, P, P, P, P]),
        "radix_lock_batch": (ctypes.c_int, [P, P, I32]),
        "radix_unlock_batch": (ctypes.c_int, [P, P, I32]),
        "radix_stats": (ctypes.c_int, [P, P]),
        "radix_check": (ctypes.c_int, [P]),
        "radix_shared_groups": (ctypes.c_int, [P, P, I32, I64, P, P, P]),
        "rx_step_stage_bytes": (SZ, [I32, I64]),
        "rx_step_plan": (ctypes.c_int, [P, I32, P, P, P, I32, I32, I64, P, SZ, P, P]),
        "rx_step_finish": (ctypes.c_int, [P, I32, P, P, P, P, P, I64, P]),
        "rx_step_workspace_bytes": (SZ, [P, P, I32]),
        "rx_step_launch": (ctypes.c_int, [P, P, P, P, P, P, P, P, I64, P, P]),
        "rx_step_run": (ctypes.c_int, [P]),
        "rx_step_prefetch": (ctypes.c_int, [P, I32, P, P, P]),
        "rx_step_ranges": (ctypes.c_int, [P, I32, P, I32, P, I32, P]),
        "rx_stage_wait": (ctypes.c_int, [P]),
        "kv_pool_write": (ctypes.c_int, [P, I32, P, P, P, P, P, P, P, P, P, I64, I64, P, P]),
        "prefix_extend_attention": (ctypes.c_int, [P, I32, P, P, P, P, I64, P, P, P, P, I32, P, P, SZ, P, P]),
        "extend_workspace_bytes": (SZ, [P, I32, I32, P]),
        "decode_workspace_bytes": (SZ, [P, I32, I32, P]),
        "decode_attention": (ctypes.c_int, [P, I32, P, P, I64, P, P, P, P, P, P, I32, P, SZ, P, P]),
        "decode_attention_noalloc": (ctypes.c_int, [P, I32, P, P, I64, P, P, P, P, P, P, I32, P, P]),
        "rx_last_error": (ctypes.c_char_p, []),
        "rx_version": (ctypes.c_char_p, []),
        "rx_wait_selftest": (ctypes.c_int, [P, U64, P]),
        "rx_set_tracing": (ctypes.c_int, [ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != RX_OK:
        raise RxError(fn, rc, load().rx_last_error().decode())


def _np_i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _addr(a: np.ndarray) -> int:
    """Host address of a contiguous numpy array.  Through a ctypes view of its buffer: about a
    third of the cost of `_addr(a)` per call, which adds up on the per-step calls (the
    array's own `ctypes` path for read-only arrays, which cannot be viewed that way)."""
    try:
        return ctypes.addressof(ctypes.c_char.from_buffer(a))
    except (TypeError, ValueError):
        return a.ctypes.data


def _ptr(t):
    """Device pointer of a tensor, or an integer device address (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    assert t.is_cuda and t.is_contiguous(), "device buffers must be contiguous CUDA tensors"
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def version() -> str:
    return load().rx_version().decode()


def set_tracing(on: bool) -> bool:
    """NVTX ranges around the library's calls (off by default); returns the previous setting."""
    return bool(load().rx_set_tracing(1 if on else 0))


def make_desc(dtype: int, hq: int, hkv: int, head_dim: int, num_slots: int, scale: float) -> rx_attn_desc:
    return rx_attn_desc(dtype, hq, hkv, head_dim, num_slots, scale)


# ============================================================================ radix tree
def radix_create(num_slots: int, slot_perm_seed: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check("radix_create", load().radix_create(num_slots, slot_perm_seed & (2 ** 64 - 1), ctypes.byref(h)))
    return h


def radix_destroy(tree) -> None:
    load().radix_destroy(tree)


def match_prefix(tree, tokens):
    """Returns (slots int32 [len], len, last node handle)."""
    tok = _np_i32(tokens)
    out = np.empty(max(len(tok), 1), np.int32)
    n, last = I64(), I64()
    _check("match_prefix", load().match_prefix(tree, _addr(tok), len(tok), _addr(out),
                                               ctypes.byref(n), ctypes.byref(last)))
    return out[: n.value].copy(), n.value, last.value


def match_prefix_len(tree, tokens) -> int:
    """Length of the longest cached prefix, without touching the tree (no stamp, no split)."""
    tok = _np_i32(tokens)
    n = I64()
    _check("match_prefix_len", load().match_prefix_len(tree, _addr(tok), len(tok), ctypes.byref(n)))
    return n.value


def match_prefix_len_batch(tree, tokens, tok_indptr) -> np.ndarray:
    tok = _np_i32(tokens)
    ind = np.ascontiguousarray(np.asarray(tok_indptr, np.int64))
    b = len(ind) - 1
    out = np.empty(max(b, 1), np.int64)
    _check("match_prefix_len_batch", load().match_prefix_len_batch(tree, b, _addr(tok), _addr(ind),
                                                                   _addr(out)))
    return out[:b].copy()


def radix_set_page_size(tree, page_size: int) -> None:
    _check("radix_set_page_size", load().radix_set_page_size(tree, page_size))


def radix_lock(tree, node: int) -> None:
    _check("radix_lock", load().radix_lock(tree, node))


def radix_unlock(tree, node: int) -> None:
    _check("radix_unlock", load().radix_unlock(tree, node))


def insert_batch_at(tree, nodes, tokens, tok_indptr, new_slots, new_indptr):
    """Insert continued from each request's matched node.  Returns (dup lengths, last nodes)."""
    nd = np.ascontiguousarray(np.asarray(nodes, np.int64))
    tok, sl = _np_i32(tokens), _np_i32(new_slots)
    ind = np.ascontiguousarray(np.asarray(tok_indptr, np.int64))
    nind = np.ascontiguousarray(np.asarray(new_indptr, np.int64))
    b = len(nd)
    dup = np.empty(max(b, 1), np.int64)
    last = np.empty(max(b, 1), np.int64)
    _check("insert_batch_at", load().insert_batch_at(tree, b, _addr(nd), _addr(tok), _addr(ind),
                                                     _addr(sl) if len(sl) else None, _addr(nind),
                                                     _addr(dup), _addr(last)))
    return dup[:b].copy(), last[:b].copy()


def radix_lock_batch(tree, nodes) -> None:
    a = np.ascontiguousarray(np.asarray(nodes, np.int64))
    _check("radix_lock_batch", load().radix_lock_batch(tree, _addr(a) if len(a) else None, len(a)))


def radix_unlock_batch(tree, nodes) -> None:
    a = np.ascontiguousarray(np.asarray(nodes, np.int64))
    _check("radix_unlock_batch", load().radix_unlock_batch(tree, _addr(a) if len(a) else None, len(a)))


def alloc_slots(tree, n: int) -> np.ndarray:
    out = np.empty(max(n, 1), np.int32)
    _check("alloc_slots", load().alloc_slots(tree, n, _addr(out)))
    return out[:n].copy()


def free_slots(tree, slots) -> None:
    s = _np_i32(slots)
    _check("free_slots", load().free_slots(tree, _addr(s) if len(s) else None, len(s)))


def insert(tree, tokens, slots):
    """Returns (dup_len, last node handle)."""
    tok, sl = _np_i32(tokens), _np_i32(slots)
    assert len(tok) == len(sl)
    dup, last = I64(), I64()
    _check("insert", load().insert(tree, _addr(tok) if len(tok) else None,
                                   _addr(sl) if len(sl) else None, len(tok),
                                   ctypes.byref(dup), ctypes.byref(last)))
    return dup.value, last.value


def evict(tree, num_tokens: int, cap: int | None = None) -> np.ndarray:
    """Frees LRU leaves until >= num_tokens are freed; returns the freed slots (the first
    `cap` of them; default: all)."""
    n = I64()
    c = radix_stats(tree)["cached_tokens"] if cap is None else cap   # at most everything cached
    out = np.empty(max(c, 1), np.int32)
    _check("evict", load().evict(tree, num_tokens, _addr(out), c, ctypes.byref(n)))
    return out[: min(n.value, c)].copy()


def evict_count(tree, num_tokens: int) -> int:
    """evict without collecting the freed slots; returns how many were freed."""
    n = I64()
    _check("evict", load().evict(tree, num_tokens, None, 0, ctypes.byref(n)))
    return n.value


def match_prefix_batch(tree, tokens, tok_indptr):
    """tokens: concatenated int32; tok_indptr int64 [batch+1].
    Returns (packed slots int32, slot indptr int64 [batch+1], last nodes int64 [batch])."""
    tok = _np_i32(tokens)
    ind = np.ascontiguousarray(np.asarray(tok_indptr, np.int64))
    b = len(ind) - 1
    out = np.empty(max(len(tok), 1), np.int32)
    oind = np.empty(b + 1, np.int64)
    last = np.empty(max(b, 1), np.int64)
    _check("match_prefix_batch", load().match_prefix_batch(tree, b, _addr(tok), _addr(ind), _addr(out),
                                                           _addr(oind), _addr(last)))
    return out[: oind[b]].copy(), oind, last[:b].copy()


def insert_batch(tree, tokens, tok_indptr, slots):
    """Returns (dup lengths int64 [batch], last nodes int64 [batch])."""
    tok, sl = _np_i32(tokens), _np_i32(slots)
    ind = np.ascontiguousarray(np.asarray(tok_indptr, np.int64))
    b = len(ind) - 1
    assert len(tok) == len(sl) == ind[b]
    dup = np.empty(max(b, 1), np.int64)
    last = np.empty(max(b, 1), np.int64)
    _check("insert_batch", load().insert_batch(tree, b, _addr(tok), _addr(ind), _addr(sl),
                                               _addr(dup), _addr(last)))
    return dup[:b].copy(), last[:b].copy()


def radix_stats(tree) -> dict:
    st = rx_stats()
    _check("radix_stats", load().radix_stats(tree, ctypes.byref(st)))
    return {f: getattr(st, f) for f, _ in rx_stats._fields_}


def radix_check(tree) -> None:
    _check("radix_check", load().radix_check(tree))


def radix_shared_groups(tree, last_nodes, min_shared: int = 1):
    """Returns (group_of int32 [batch], group_len int64 [num_groups])."""
    ln = np.ascontiguousarray(np.asarray(last_nodes, np.int64))
    b = len(ln)
    gof = np.empty(max(b, 1), np.int32)
    glen = np.empty(max(b, 1), np.int64)
    ng = I32()
    _check("radix_shared_groups", load().radix_shared_groups(tree, _addr(ln), b, min_shared, _addr(gof),
                                                             _addr(glen), ctypes.byref(ng)))
    return gof[:b].copy(), glen[: ng.value].copy()


def rx_step_stage_bytes(batch: int, total_tokens: int) -> int:
    return int(load().rx_step_stage_bytes(batch, total_tokens))


def rx_step_plan(tree, tokens: np.ndarray, tok_indptr: np.ndarray, n_new: np.ndarray, group_mode: int,
                 heads_per_kv: int, min_shared: int, stage_addr: int, stage_cap: int, out_last: np.ndarray):
    """tokens int32, tok_indptr int64 [batch+1], n_new int32 [batch], out_last int64 [batch]
    (filled): all contiguous.  stage_addr: host address of the staging buffer.  Returns the
    rx_step_layout."""
    b = len(tok_indptr) - 1
    lay = rx_step_layout()
    _check("rx_step_plan", load().rx_step_plan(
        tree, b, _addr(tokens), _addr(tok_indptr), _addr(n_new) if b else None,
        group_mode, heads_per_kv, min_shared, stage_addr, stage_cap, _addr(out_last) if b else None,
        ctypes.byref(lay)))
    return lay


def rx_step_finish(tree, tokens: np.ndarray, tok_indptr: np.ndarray, last_nodes: np.ndarray, stage_addr: int,
                   layout, evict_tokens: int) -> int:
    """Returns the number of slots evicted."""
    n = I64()
    _check("rx_step_finish", load().rx_step_finish(
        tree, layout.batch, _addr(tokens), _addr(tok_indptr),
        _addr(last_nodes) if layout.batch else None, stage_addr, ctypes.byref(layout), evict_tokens,
        ctypes.byref(n)))
    return n.value


def rx_step_workspace_bytes(desc, layout, decode: bool) -> int:
    return int(load().rx_step_workspace_bytes(ctypes.byref(desc), ctypes.byref(layout), 1 if decode else 0))


def rx_step_prefetch(desc, n_new: np.ndarray, io, stream) -> None:
    """Start the host-buffer copies of a step's new rows before it is planned."""
    nn = np.ascontiguousarray(np.asarray(n_new, np.int32))
    _check("rx_step_prefetch", load().rx_step_prefetch(ctypes.byref(desc), len(nn), _addr(nn) if len(nn) else None,
                                                       ctypes.byref(io), _stream(stream)))


def rx_step_ranges(desc, n_new: np.ndarray, chunks: int = 0) -> np.ndarray:
    """The request cut points (first 0, last batch) of a host-buffer step's copy pipeline."""
    nn = np.ascontiguousarray(np.asarray(n_new, np.int32))
    cap = max(int(chunks), 4) + 2
    cuts = np.zeros(cap, np.int32)
    n = ctypes.c_int32(0)
    _check("rx_step_ranges", load().rx_step_ranges(ctypes.byref(desc), len(nn), _addr(nn) if len(nn) else None,
                                                   int(chunks), _addr(cuts), cap, ctypes.byref(n)))
    return cuts[: n.value + 1].copy()


def rx_step_launch(tree, desc, tokens: np.ndarray, tok_indptr: np.ndarray, last_nodes: np.ndarray, stage_addr: int,
                   layout, io, evict_tokens: int, stream) -> int:
    """Copy, kv_pool_write, attention and finish of a planned step in one call; returns the
    number of slots evicted."""
    n = I64()
    _check("rx_step_launch", load().rx_step_launch(
        tree, ctypes.byref(desc), _addr(tokens), _addr(tok_indptr),
        _addr(last_nodes) if layout.batch else None, stage_addr, ctypes.byref(layout), ctypes.byref(io),
        evict_tokens, ctypes.byref(n), _stream(stream)))
    return n.value


def rx_step_run(args) -> int:
    """Plan and launch a step in one call.  args: an rx_step_args (tokens int32, tok_indptr
    int64, n_new int32, out_last int64 [batch]: host addresses of contiguous arrays; out: the
    address of an rx_step_layout to fill), or its address as an int.  Returns RX_OK, or
    RX_ENOMEM when io's device buffers are too small for the plan (planned and pinned, not
    launched: grow them and call rx_step_launch); raises otherwise."""
    rc = load().rx_step_run(args if isinstance(args, int) else ctypes.addressof(args))
    if rc != RX_OK and rc != RX_ENOMEM:
        _check("rx_step_run", rc)
    return rc


_step_ext = None


def step_ext():
    """The _rxstep extension (the per-step marshalling of rx_step_run in C, built next to the
    library where the Python headers are installed), bound to the loaded library's rx_step_run;
    None when it was not built (the ctypes path then makes the same call)."""
    global _step_ext
    if _step_ext is None:
        from .build import pystep_path
        path = pystep_path()
        _step_ext = False
        if os.path.exists(path):
            import importlib.machinery
            import importlib.util
            loader = importlib.machinery.ExtensionFileLoader("_rxstep", path)
            spec = importlib.util.spec_from_file_location("_rxstep", path, loader=loader)
            m = importlib.util.module_from_spec(spec)
            loader.exec_module(m)
            m.bind(ctypes.cast(load().rx_step_run, ctypes.c_void_p).value)
            _step_ext = m
    return _step_ext or None


def rx_wait_selftest(status, limit_ns: int, stream=None) -> None:
    """The kernels' bounded wait run out on purpose (a barrier nobody arrives at): *status
    becomes RX_DEV_TIMEOUT once the stream reaches it (see include/radix_attn.h)."""
    _check("rx_wait_selftest", load().rx_wait_selftest(_ptr(status), int(limit_ns), _stream(stream)))


def rx_stage_wait(stage_addr: int) -> None:
    _check("rx_stage_wait", load().rx_stage_wait(stage_addr))


class RadixTree:
    """Owning wrapper of an rx_radix handle."""

    def __init__(self, num_slots: int, seed: int, page_size: int = 1):
        self.h = radix_create(num_slots, seed)
        self.num_slots = num_slots
        self.page_size = page_size
        if page_size != 1:
            radix_set_page_size(self.h, page_size)

    def __del__(self):
        if getattr(self, "h", None) is not None and _lib is not None:
            radix_destroy(self.h)
            self.h = None

    def match_prefix(self, tokens):
        return match_prefix(self.h, tokens)

    def insert(self, tokens, slots):
        return insert(self.h, tokens, slots)

    def match_prefix_len(self, tokens):
        return match_prefix_len(self.h, tokens)

    def match_prefix_len_batch(self, tokens, tok_indptr):
        return match_prefix_len_batch(self.h, tokens, tok_indptr)

    def evict(self, n, cap=None):
        return evict(self.h, n, cap)

    def evict_count(self, n):
        return evict_count(self.h, n)

    def alloc_slots(self, n):
        return alloc_slots(self.h, n)

    def free_slots(self, slots):
        return free_slots(self.h, slots)

    def lock(self, node):
        return radix_lock(self.h, node)

    def unlock(self, node):
        return radix_unlock(self.h, node)

    def match_prefix_batch(self, tokens, tok_indptr):
        return match_prefix_batch(self.h, tokens, tok_indptr)

    def insert_batch(self, tokens, tok_indptr, slots):
        return insert_batch(self.h, tokens, tok_indptr, slots)

    def insert_batch_at(self, nodes, tokens, tok_indptr, new_slots, new_indptr):
        return insert_batch_at(self.h, nodes, tokens, tok_indptr, new_slots, new_indptr)

    def lock_batch(self, nodes):
        return radix_lock_batch(self.h, nodes)

    def unlock_batch(self, nodes):
        return radix_unlock_batch(self.h, nodes)

    def stats(self):
        return radix_stats(self.h)

    def check(self):
        return radix_check(self.h)

    def shared_groups(self, last_nodes, min_shared=1):
        return radix_shared_groups(self.h, last_nodes, min_shared)


# ============================================================================ kernels
def kv_pool_write(desc, batch, prefix_slots, prefix_indptr, new_slots, qo_indptr, k_new, v_new, k_pool, v_pool,
                  req_to_token, total_new, status, stream=None, r2t_stride=None) -> None:
    """req_to_token: a [batch, stride] tensor, or a device address with r2t_stride given."""
    stride = req_to_token.shape[1] if r2t_stride is None else r2t_stride
    _check("kv_pool_write", load().kv_pool_write(
        ctypes.byref(desc), batch, _ptr(prefix_slots), _ptr(prefix_indptr), _ptr(new_slots), _ptr(qo_indptr),
        _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(req_to_token), stride,
        total_new, _ptr(status), _stream(stream)))


def prefix_extend_attention(desc, batch, q, qo_indptr, prefix_lens, req_to_token, k_pool, v_pool, out, lse,
                            max_qo_len, status, groups=None, workspace=None, stream=None, r2t_stride=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    stride = req_to_token.shape[1] if r2t_stride is None else r2t_stride
    _check("prefix_extend_attention", load().prefix_extend_attention(
        ctypes.byref(desc), batch, _ptr(q), _ptr(qo_indptr), _ptr(prefix_lens), _ptr(req_to_token),
        stride, _ptr(k_pool), _ptr(v_pool), _ptr(out), _ptr(lse), max_qo_len,
        ctypes.byref(groups) if groups is not None else None, _ptr(workspace), ws_bytes, _ptr(status),
        _stream(stream)))


def extend_workspace_bytes(desc, batch, max_qo_len, groups=None) -> int:
    return int(load().extend_workspace_bytes(ctypes.byref(desc), batch, max_qo_len,
                                             ctypes.byref(groups) if groups is not None else None))


def shared_groups_struct(num_groups, max_group_size, group_indptr, group_members, group_len, max_group_len,
                         max_group_rows=0):
    """rx_shared_groups from device int32 arrays (tensors or device addresses)."""
    if num_groups == 0:
        return None
    return rx_shared_groups(num_groups, max_group_size, _ptr(group_indptr), _ptr(group_members),
                            _ptr(group_len), max_group_len, max_group_rows)


def decode_workspace_bytes(desc, batch, max_kv_len, groups=None) -> int:
    return int(load().decode_workspace_bytes(ctypes.byref(desc), batch, max_kv_len,
                                             ctypes.byref(groups) if groups is not None else None))


def decode_attention(desc, batch, q, req_to_token, kv_lens, k_pool, v_pool, out, lse, max_kv_len, workspace,
                     status, groups=None, stream=None, r2t_stride=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    stride = req_to_token.shape[1] if r2t_stride is None else r2t_stride
    _check("decode_attention", load().decode_attention(
        ctypes.byref(desc), batch, _ptr(q), _ptr(req_to_token), stride, _ptr(kv_lens),
        ctypes.byref(groups) if groups is not None else None, _ptr(k_pool), _ptr(v_pool), _ptr(out), _ptr(lse),
        max_kv_len, _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)))


def decode_attention_noalloc(desc, batch, q, req_to_token, kv_lens, k_pool, v_pool, out, lse, max_kv_len, status,
                             groups=None, stream=None, r2t_stride=None) -> None:
    """decode_attention with the library's static scratch instead of a workspace: for callers
    that cannot allocate device memory per call.  Overlapping calls race (one shared array).
    req_to_token is a [batch, stride] tensor, or a device address with r2t_stride given."""
    stride = req_to_token.shape[1] if r2t_stride is None else r2t_stride
    _check("decode_attention_noalloc", load().decode_attention_noalloc(
        ctypes.byref(desc), batch, _ptr(q), _ptr(req_to_token), stride, _ptr(kv_lens),
        ctypes.byref(groups) if groups is not None else None, _ptr(k_pool), _ptr(v_pool), _ptr(out), _ptr(lse),
        max_kv_len, _ptr(status), _stream(stream)))
