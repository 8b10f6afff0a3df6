"""One attention layer's prefix cache on one GPU: radix tree + KV pools + kernels.

A step over a batch of requests (each a full prompt whose tail is new):
  a1 match_prefix_batch (host tree)   -> matched slots and lengths P_b
  a2 alloc_slots (host allocator)     -> slots for the n_b new tokens
  a3 kv_pool_write (CUDA)             -> req_to_token table, new K/V scattered into the pools
  a4 prefix_extend_attention (CUDA)   or  a5/a6 decode_attention (CUDA, split-KV + merge)
  a7 insert_batch (host tree)         -> the new tokens become cached
  a8 evict (host tree)                -> LRU leaves freed under memory pressure
"SGLang: Efficient Execution of Structured Language Model Programs" (RadixAttention) and
"Prompt Caching" (Ultralytics glossary, "How prompt caching works").  This module only
strings library calls together and moves the step's small index arrays to the device.
"""
from __future__ import annotations


import ctypes

import numpy as np
import torch

from . import api


def _dev_from_host(a, dtype_bits, device):
    """Host numpy array -> device tensor; bf16 arrives as uint16 bit patterns."""
    if dtype_bits == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device, non_blocking=False)


_DTYPES = {np.int32: np.dtype(np.int32), np.int64: np.dtype(np.int64)}


def _contig(a, dt):
    """a as a C-contiguous array of dtype dt (the array itself when it already is one)."""
    if type(a) is np.ndarray and a.dtype is _DTYPES.get(dt) and a.flags.c_contiguous:
        return a
    return np.ascontiguousarray(a, dt)


class StepPlan:
    """One planned step.  The index arrays are views of the pinned staging buffer the step's
    device copy is made from (two buffers alternate: a plan stays valid until the plan after
    next); each is made on first use."""
    __slots__ = ("batch", "tokens", "tok_indptr", "last_nodes", "layout", "stage", "_host", "_views")

    def __init__(self, batch, tokens, tok_indptr, last_nodes, layout, stage, host):
        self.batch = batch
        self.tokens = tokens            # concatenated full prompts (cached part + new tokens)
        self.tok_indptr = tok_indptr    # [batch+1]
        self.last_nodes = last_nodes    # [batch] node where each match ended (pinned until finish)
        self.layout = layout            # rx_step_layout of the staging buffer
        self.stage = stage              # which staging buffer
        self._host = host
        self._views = None

    @property
    def max_qo_len(self):
        return self.layout.max_qo_len

    @property
    def max_kv_len(self):
        return self.layout.max_kv_len

    @property
    def stride(self):
        return self.layout.stride

    def _view(self, name, off, n, dt):
        if self._views is None:
            self._views = {}
        v = self._views.get(name)
        if v is None:
            v = self._views[name] = self._host[off:off + n * np.dtype(dt).itemsize].view(dt)
        return v

    @property
    def prefix_slots(self):             # packed matched slots
        L = self.layout
        return self._view("ps", L.off_prefix_slots, L.total_prefix, np.int32)

    @property
    def prefix_indptr(self):            # [batch+1]
        return self._view("pi", self.layout.off_prefix_indptr, self.batch + 1, np.int64)

    @property
    def prefix_lens(self):              # [batch] int32 (P_b)
        return self._view("pl", self.layout.off_prefix_lens, self.batch, np.int32)

    @property
    def new_slots(self):                # [T]
        L = self.layout
        return self._view("ns", L.off_new_slots, L.total_new, np.int32)

    @property
    def qo_indptr(self):                # [batch+1]
        return self._view("qo", self.layout.off_qo_indptr, self.batch + 1, np.int64)

    @property
    def grp_indptr(self):               # shared-prefix groups (None without)
        L = self.layout
        return self._view("gi", L.off_grp_indptr, L.num_groups + 1, np.int32) if L.num_groups else None

    @property
    def grp_members(self):
        L = self.layout
        return self._view("gm", L.off_grp_members, int(self.grp_indptr[-1]), np.int32) if L.num_groups else None

    @property
    def grp_len(self):
        L = self.layout
        return self._view("gl", L.off_grp_len, L.num_groups, np.int32) if L.num_groups else None

    @property
    def grp_rows(self):                 # largest sum of new tokens over a group's members
        return self.layout.max_group_rows if self.layout.num_groups else 0


_GROUP_MODE = {False: api.RX_GROUPS_NONE, None: api.RX_GROUPS_NONE, True: api.RX_GROUPS_ALWAYS,
               "auto": api.RX_GROUPS_AUTO}


class PrefixCacheEngine:
    def __init__(self, dtype: str, hq: int, hkv: int, head_dim: int, num_slots: int, seed: int,
                 device: str = "cuda", poison: bool = True, num_layers: int = 1, page_size: int = 1):
        """One radix tree over `num_layers` layers' KV pools: a cached token has one slot, and
        every layer keeps that token's K/V at the same slot of its own pool (the tree, the
        plan, the slot table and the index upload are shared by the layers of a step)."""
        self.dtype = dtype
        self.tdtype = torch.float32 if dtype == "f32" else torch.bfloat16
        self.hq, self.hkv, self.d = hq, hkv, head_dim
        self.num_slots = num_slots
        self.device = torch.device(device)
        self.tree = api.RadixTree(num_slots, seed, page_size=page_size)
        self.num_layers = num_layers
        self.k_pools = torch.empty(num_layers, num_slots, hkv, head_dim, dtype=self.tdtype, device=self.device)
        self.v_pools = torch.empty_like(self.k_pools)
        if poison:   # unused slots hold NaN so that any stray gather shows up
            self.k_pools.fill_(float("nan"))
            self.v_pools.fill_(float("nan"))
        self.k_pool, self.v_pool = self.k_pools[0], self.v_pools[0]   # layer 0 (single-layer use)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.desc = api.make_desc(api.RX_F32 if dtype == "f32" else api.RX_BF16, hq, hkv, head_dim, num_slots,
                                  1.0 / float(np.sqrt(head_dim)))
        self._ws = None
        # step index arrays travel in one pinned buffer (two, alternating) and one H2D copy
        self._pin = [None, None]        # pinned host staging (torch tensor, numpy view, address)
        self._pin_np = [None, None]
        self._pin_addr = [0, 0]
        self._io_static = None          # the io whose buffer addresses are current
        self._ws_need = {}
        self._pin_ev = [torch.cuda.Event(), torch.cuda.Event()]
        self._pin_used = [False, False]
        self._pin_i = 0
        self._dev_idx = None
        self._dev_stage = [None, None]  # the one-call path's device copies of the staging buffers
        self._r2t = None
        self._r2t_flat = None     # the one-call path's slot table ([batch, stride] in a flat buffer)
        self._last = [None, None]  # the one-call path's match-end nodes, per staging buffer
        self._args = [None, None]  # the one-call path's rx_step_args and layout, per staging buffer
        self._args_addr = [0, 0]
        self._args_set = [None, None]  # the per-buffer fields last written into each
        self._layout = [None, None]
        self._dev_stage_cap = [0, 0]
        self._dev_stage_ptr = [0, 0]
        self._io_addr = 0
        self._stream_handle = 0
        self._ext = None
        self._bound_bufs = (None, None)  # the slot table and workspace objects bound into the io
        self._io_flags = None            # (overlap, decode) last written into the io
        self._io_host = False            # the io holds host-buffer addresses
        self._io = None
        self._stage_need = {}     # (batch, total tokens) -> staging bytes
        self._stream = torch.cuda.current_stream(self.device)

    # ------------------------------------------------------------------ helpers
    def _i32(self, a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(self.device)

    def _i64(self, a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(self.device)

    def device_status(self) -> int:
        return int(self.status.item())

    # ------------------------------------------------------------------ cached history
    def populate(self, tokens: np.ndarray, k, v) -> int:
        """Cache one earlier sequence: match, allocate the uncached tail, write its K/V,
        insert.  k, v: [len, hkv, d] for the whole sequence (host arrays or device tensors),
        or lists of those, one per layer.  Returns the number of tokens newly written."""
        tokens = np.ascontiguousarray(tokens, np.int32)
        slots, m, _ = self.tree.match_prefix(tokens)
        n = len(tokens) - m
        if n == 0:
            return 0
        new = self.tree.alloc_slots(n)
        ks = k if isinstance(k, (list, tuple)) else [k]
        vs = v if isinstance(v, (list, tuple)) else [v]
        assert len(ks) == len(vs) <= self.num_layers
        r2t = torch.empty(1, len(tokens), dtype=torch.int32, device=self.device)
        ps, pi, ns, qi = self._i32(slots if m else [0]), self._i64([0, m]), self._i32(new), self._i64([0, n])
        for layer, (kl, vl) in enumerate(zip(ks, vs)):
            kn = kl[m:] if isinstance(kl, torch.Tensor) else _dev_from_host(kl[m:], self.dtype, self.device)
            vn = vl[m:] if isinstance(vl, torch.Tensor) else _dev_from_host(vl[m:], self.dtype, self.device)
            api.kv_pool_write(self.desc, 1, ps, pi, ns, qi, kn.contiguous(), vn.contiguous(), self.k_pools[layer],
                              self.v_pools[layer], r2t, n, self.status)
        dup, _ = self.tree.insert(tokens, np.concatenate([slots, new]))
        if dup > m:
            self.tree.free_slots(new[: dup - m])
        return n

    # ------------------------------------------------------------------ step
    def new_token_counts(self, prompts) -> np.ndarray:
        """How many trailing tokens of each prompt must be computed now: those past its
        reusable cached prefix (whole pages only when the tree has a page size above one)."""
        if not len(prompts):
            return np.zeros(0, np.int64)
        ind = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int64)
        m = self.tree.match_prefix_len_batch(np.concatenate(prompts).astype(np.int32), ind)
        return np.diff(ind) - m

    def plan(self, prompts, n_new, groups: bool = False, min_shared: int = 64) -> StepPlan:
        """a1 + a2 for a list of prompts (see plan_concat)."""
        b = len(prompts)
        lens = np.array([len(p) for p in prompts], np.int64)
        tok_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        tokens = np.concatenate(prompts).astype(np.int32) if b else np.zeros(0, np.int32)
        return self.plan_concat(tokens, tok_indptr, n_new, groups, min_shared)

    def _staging(self, nbytes: int, native_wait: bool = True) -> int:
        """Next pinned staging buffer with room for nbytes, once the copy that last read it is done
        (native_wait=False: the caller's native call waits for a native step's copy itself, unless
        the buffer has to be replaced here)."""
        i = self._pin_i
        self._pin_i ^= 1
        if self._pin[i] is not None and (native_wait or self._pin[i].numel() < nbytes):
            api.rx_stage_wait(self._pin_addr[i])            # a native step's copy out of it is done
        if self._pin[i] is None or self._pin[i].numel() < nbytes:
            if self._pin_used[i]:
                self._pin_ev[i].synchronize()
            self._pin[i] = torch.empty(max(nbytes, 4096) * 2, dtype=torch.uint8).pin_memory()
            self._pin_np[i] = self._pin[i].numpy()
            self._pin_addr[i] = self._pin[i].data_ptr()
            self._pin_used[i] = False
        if self._pin_used[i]:
            self._pin_ev[i].synchronize()
            self._pin_used[i] = False
        return i

    def plan_concat(self, tokens, tok_indptr, n_new, groups=False, min_shared: int = 64) -> StepPlan:
        """a1 + a2: match every prompt (tokens[tok_indptr[b]:tok_indptr[b+1]]), check that
        exactly its last n_new[b] tokens are uncached, allocate their slots, pin the matched
        prefixes until finish; with groups (True, or "auto": only where stacking pays) the
        shared-prefix groups too.  All in the library (rx_step_plan), written straight into a
        pinned staging buffer."""
        tokens = _contig(tokens, np.int32)
        tok_indptr = _contig(tok_indptr, np.int64)
        n_new = _contig(n_new, np.int32)
        b = len(tok_indptr) - 1
        key = (b, int(tok_indptr[-1]))
        need = self._stage_need.get(key)
        if need is None:
            need = self._stage_need[key] = api.rx_step_stage_bytes(*key)
        i = self._staging(need)
        host = self._pin_np[i]
        last = np.empty(max(b, 1), np.int64)
        L = api.rx_step_plan(self.tree.h, tokens, tok_indptr, n_new, _GROUP_MODE[groups], self.hq // self.hkv,
                             min_shared, self._pin_addr[i], host.nbytes, last)
        return StepPlan(b, tokens, tok_indptr, last[:b], L, i, host)

    def step(self, tokens, tok_indptr, n_new, q, k_new, v_new, out, lse=None, decode: bool = False,
             groups=False, min_shared: int = 64, evict_tokens: int = 0, stream=None, host=None,
             chunks: int = 0, overlap: bool = False) -> StepPlan:
        """A whole step in one library call, rx_step_run: rx_step_plan (a1, a2, groups, pinning,
        into a pinned staging buffer) then rx_step_launch (the index arrays to the device, a3,
        a4 or a5/a6, then a7/a8 and unpinning).  q/k_new/v_new are the step's new rows in request
        order; out receives the attention output.  With host=(q_h, k_h, v_h, out_h[, lse_h])
        (pinned host tensors of the same shapes) the rows come from and the output goes to host
        memory, copied by the library as a pipeline of `chunks` request ranges (0: automatic):
        the input copies start before the plan is made (inside the same call) and run behind the
        kernels with the output copies; they are complete when the stream is.  overlap=True: in
        host mode the input copies wait only for the kernels of the last step that read the same
        q buffer, not for all work on the stream -- with two sets of device rows used in turn, a
        step's copies run under the previous step's kernels (nothing else may still read
        q/k_new/v_new); with device rows the index arrays' copy runs on a copy stream under the
        previous step's kernels (the engine alternates two device copies of the staging buffer).
        When a device buffer turns out too small for the plan, it is grown and the planned step
        launched with rx_step_launch.  Returns the plan (its index arrays stay readable until the
        plan after next)."""
        io = self._io
        if io is None:
            io = self._io = api.rx_step_io()
            self._io_addr = ctypes.addressof(io)
            self._stream_handle = self._stream.cuda_stream
            self._ext = api.step_ext()
        if host is not None:
            io.h_q, io.h_k_new, io.h_v_new, io.h_out = (x.data_ptr() for x in host[:4])
            io.h_lse = host[4].data_ptr() if len(host) > 4 and host[4] is not None else None
            io.chunks = int(chunks)
            self._io_host = True
        elif self._io_host:
            io.h_q = io.h_k_new = io.h_v_new = io.h_out = io.h_lse = None
            io.chunks = 0
            self._io_host = False
        flags = (1 if overlap else 0, 1 if decode else 0)
        if flags != self._io_flags:
            io.overlap, io.decode = flags
            self._io_flags = flags
        tokens = _contig(tokens, np.int32)
        tok_indptr = _contig(tok_indptr, np.int64)
        n_new = _contig(n_new, np.int32)
        b = len(tok_indptr) - 1
        key = (b, int(tok_indptr[-1]))
        need = self._stage_need.get(key)
        if need is None:
            need = self._stage_need[key] = api.rx_step_stage_bytes(*key)
        i = self._pin_i
        if self._pin[i] is not None and not self._pin_used[i] and self._pin_np[i].nbytes >= need:
            self._pin_i = i ^ 1           # the buffer fits; the library waits for its last reader
        else:
            i = self._staging(need, native_wait=False)
        hbuf = self._pin_np[i]
        # the device copy of the index arrays alternates with the pinned staging buffer, so that
        # with overlap a step's copy can run while the previous step's kernels read the other;
        # the plan's arrays never take more than the staging buffer's bound
        if self._dev_stage_cap[i] < need:
            ds = self._dev_stage[i] = torch.empty(max(need, 4096) * 2, dtype=torch.uint8, device=self.device)
            self._dev_stage_cap[i], self._dev_stage_ptr[i] = ds.numel(), ds.data_ptr()
        if self._r2t_flat is None:
            self._r2t_flat = torch.empty(max(b, 1) * 1024, dtype=torch.int32, device=self.device)
        # rebind when a buffer was replaced (here, or the workspace by a per-operation call)
        if self._io_static is not io or self._bound_bufs[0] is not self._r2t_flat or self._bound_bufs[1] is not self._ws:
            self._bind_io(io)
        a = self._args[i]
        if a is None:
            a = self._args[i] = api.rx_step_args()
            self._args_addr[i] = ctypes.addressof(a)
            L = self._layout[i] = api.rx_step_layout()
            a.tree, a.desc, a.io, a.out = self.tree.h, ctypes.addressof(self.desc), ctypes.addressof(io), \
                ctypes.addressof(L)
        L = self._layout[i]
        last = self._last[i]
        if last is None or len(last) < max(b, 1):
            last = self._last[i] = np.empty(max(b, 1) * 2, np.int64)
            a.out_last = api._addr(last)
        # the struct's per-buffer fields, only when they change
        per = (_GROUP_MODE[groups], min_shared, evict_tokens,
               self._stream_handle if stream is None else api._stream(stream), self._pin_addr[i], hbuf.nbytes)
        if per != self._args_set[i]:
            a.group_mode, a.heads_per_kv, a.min_shared, a.evict_tokens = per[0], self.hq // self.hkv, per[1], per[2]
            a.stream, a.h_stage, a.stage_cap = per[3], per[4], per[5]
            self._args_set[i] = per
        # the step's inputs (and the device staging copy that goes with this buffer), and the call
        ext = self._ext
        if ext is not None:
            rc = ext.run(self._args_addr[i], self._io_addr, b, tokens, tok_indptr, n_new, q, k_new, v_new, out, lse,
                         self._dev_stage_ptr[i], self._dev_stage_cap[i])
            if rc != api.RX_OK and rc != api.RX_ENOMEM:
                api._check("rx_step_run", rc)
        else:
            io.d_stage, io.d_stage_bytes = self._dev_stage_ptr[i], self._dev_stage_cap[i]
            io.d_q, io.d_k_new, io.d_v_new = q.data_ptr(), k_new.data_ptr(), v_new.data_ptr()
            io.d_out, io.d_lse = out.data_ptr(), (lse.data_ptr() if lse is not None else None)
            a.batch, a.tokens, a.tok_indptr, a.n_new = b, api._addr(tokens), api._addr(tok_indptr), api._addr(n_new)
            rc = api.rx_step_run(self._args_addr[i])
        if rc == api.RX_ENOMEM:
            # planned and pinned, not launched: grow the slot table or the workspace, then launch
            r2t_need = max(L.batch, 1) * L.stride
            if self._r2t_flat.numel() < r2t_need:
                self._r2t_flat = torch.empty(r2t_need * 2, dtype=torch.int32, device=self.device)
            wkey = (decode, L.batch, L.max_qo_len, L.max_kv_len, L.num_groups, L.max_group_size, L.max_group_len,
                    L.max_group_rows)
            ws_need = self._ws_need.get(wkey)
            if ws_need is None:
                ws_need = self._ws_need[wkey] = api.rx_step_workspace_bytes(self.desc, L, decode)
            if ws_need and (self._ws is None or self._ws.numel() < ws_need):
                self._ws = torch.empty(ws_need, dtype=torch.uint8, device=self.device)
            self._bind_io(io)
            api.rx_step_launch(self.tree.h, self.desc, tokens, tok_indptr, last, self._pin_addr[i], L, io,
                               evict_tokens, self._stream_handle if stream is None else api._stream(stream))
        return StepPlan(b, tokens, tok_indptr, last[:b], L, i, hbuf)

    def _bind_io(self, io) -> None:
        """The step io's long-lived buffer addresses (pools, slot table, workspace, status)."""
        io.d_k_pool, io.d_v_pool = self.k_pool.data_ptr(), self.v_pool.data_ptr()
        io.d_r2t, io.r2t_elems = self._r2t_flat.data_ptr(), self._r2t_flat.numel()
        io.d_workspace = self._ws.data_ptr() if self._ws is not None else None
        io.ws_bytes = self._ws.numel() if self._ws is not None else 0
        io.d_status = self.status.data_ptr()
        self._io_static = io
        self._bound_bufs = (self._r2t_flat, self._ws)

    def upload(self, plan: StepPlan, stream=None) -> dict:
        """Move the step's index arrays to the device: one asynchronous H2D copy of the staging
        buffer on the stream.  Returns device addresses (same offsets as the staging buffer)."""
        L, i = plan.layout, plan.stage
        total = max(int(L.bytes), 256)
        if self._dev_idx is None or self._dev_idx.numel() < total:
            self._dev_idx = torch.empty(max(total, 4096) * 2, dtype=torch.uint8, device=self.device)
        st = self._stream if stream is None else stream
        with torch.cuda.stream(st):
            self._dev_idx[:total].copy_(self._pin[i][:total], non_blocking=True)
        self._pin_ev[i].record(st)
        self._pin_used[i] = True
        base = self._dev_idx.data_ptr()
        out = {"prefix_slots": base + L.off_prefix_slots, "prefix_indptr": base + L.off_prefix_indptr,
               "new_slots": base + L.off_new_slots, "qo_indptr": base + L.off_qo_indptr,
               "prefix_lens": base + L.off_prefix_lens, "kv_lens": base + L.off_kv_lens}
        if L.num_groups:
            out.update(grp_indptr=base + L.off_grp_indptr, grp_members=base + L.off_grp_members,
                       grp_len=base + L.off_grp_len)
        B = plan.batch
        if self._r2t is None or self._r2t.shape[1] != plan.stride or self._r2t.shape[0] < max(B, 1):
            self._r2t = torch.empty(max(B, 1) * 2, plan.stride, dtype=torch.int32, device=self.device)
        out["r2t"] = self._r2t
        out["batch"] = B
        out["stride"] = plan.stride
        return out

    def write(self, plan: StepPlan, dev: dict, k_new, v_new, stream=None, layer: int = 0) -> None:
        """a3: slot table + scatter of the new tokens' K/V into `layer`'s pools."""
        api.kv_pool_write(self.desc, plan.batch, dev["prefix_slots"], dev["prefix_indptr"], dev["new_slots"],
                          dev["qo_indptr"], k_new, v_new, self.k_pools[layer], self.v_pools[layer], dev["r2t"],
                          int(plan.qo_indptr[-1]), self.status, stream or self._stream.cuda_stream)

    def extend(self, plan: StepPlan, dev: dict, q, out, lse=None, stream=None, layer: int = 0) -> None:
        """a4: new tokens attend to their cached prefix and causally to themselves (with the
        plan's shared-prefix groups, if any: shared run once per group, stacked rows)."""
        grp = self.groups(plan, dev)
        ws = None
        if grp is not None:
            nbytes = api.extend_workspace_bytes(self.desc, plan.batch, plan.max_qo_len, grp)
            if self._ws is None or self._ws.numel() < nbytes:
                self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            ws = self._ws
        api.prefix_extend_attention(self.desc, plan.batch, q, dev["qo_indptr"], dev["prefix_lens"], dev["r2t"],
                                    self.k_pools[layer], self.v_pools[layer], out, lse, plan.max_qo_len, self.status,
                                    groups=grp, workspace=ws, stream=stream or self._stream.cuda_stream)

    def groups(self, plan: StepPlan, dev: dict):
        """The plan's shared-prefix groups (computed by plan(..., groups=True) and uploaded with
        the step's index arrays) as the ABI struct, or None."""
        L = plan.layout
        if not L.num_groups:
            return None
        return api.shared_groups_struct(L.num_groups, L.max_group_size, dev["grp_indptr"], dev["grp_members"],
                                        dev["grp_len"], L.max_group_len, L.max_group_rows)

    def decode_workspace(self, plan: StepPlan, groups=None):
        nbytes = api.decode_workspace_bytes(self.desc, plan.batch, plan.max_kv_len, groups)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def decode(self, plan: StepPlan, dev: dict, q, out, lse=None, groups=None, stream=None, layer: int = 0) -> None:
        """a5 + a6: one query token per request over all of its cached tokens."""
        ws = self.decode_workspace(plan, groups)
        api.decode_attention(self.desc, plan.batch, q, dev["r2t"], dev["kv_lens"], self.k_pools[layer],
                             self.v_pools[layer], out,
                             lse, plan.max_kv_len, ws, self.status, groups=groups,
                             stream=stream or self._stream.cuda_stream)

    def commit(self, plan: StepPlan) -> np.ndarray:
        """a7: insert every prompt, continuing from the node its match ended at; frees new
        slots whose tokens turned out to be cached meanwhile (by an earlier request of the batch)."""
        dup, _ = self.tree.insert_batch_at(plan.last_nodes, plan.tokens, plan.tok_indptr, plan.new_slots,
                                           plan.qo_indptr)
        over = dup - plan.prefix_lens
        if (over > 0).any():
            extra = [plan.new_slots[plan.qo_indptr[b]:plan.qo_indptr[b] + over[b]] for b in np.flatnonzero(over > 0)]
            self.tree.free_slots(np.concatenate(extra))
        return dup

    def release(self, num_tokens: int) -> np.ndarray:
        """a8: evict least-recently-used unlocked leaves until num_tokens are freed."""
        return self.tree.evict(num_tokens)

    def finish(self, plan: StepPlan, evict_tokens: int = 0) -> int:
        """End of a step: a7 insert, a8 evict (the step's prefixes still pinned), unpin -- one
        library call (rx_step_finish).  Returns the number of slots evicted."""
        return api.rx_step_finish(self.tree.h, plan.tokens, plan.tok_indptr, plan.last_nodes,
                                  self._pin[plan.stage].data_ptr(), plan.layout, evict_tokens)
