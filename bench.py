"""Benchmark: prefix-cached attention steps on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload c5] [--subs c3,c4,c2]

One step is one pass of the whole hot path over one batch: host radix match and slot
allocation, upload of the step's index arrays, kv_pool_write (slot table + K/V scatter),
the attention kernel(s) (extend, or split-KV decode + merge), insert of the new tokens
and LRU eviction of as many cached tokens (so the cache stays at a steady size).  Every
step's requests carry fresh new-token ids, so each step is a new batch of requests that
hits the cached prefix.  Inputs (Q and the new K/V) are resident in HBM when the timed
region starts; the e2e figure repeats the step through the same public call with the inputs
in pinned host memory: the library copies them in and the output back inside the timed
region (a pipeline of request ranges whose copies run behind the kernels).

The headline line is the long multi-turn chat workload (c5: 32 requests x 1024 new tokens over
29,491 cached, GQA 64/8 x 128), the largest single-GPU one; the few-shot tree (c3), the batched
decode (c4), the shared system prompt (c2) and the tiny fp32 case (c1) are measured in the same
run and reported under "sub_results" with the same keys.

Prints one JSON line.  With N > 1 (torchrun) every rank runs its own replica of the
workload on its own GPU (the path shards over independent requests; no collective is
needed), value = all ranks' tokens / max over ranks of the time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "prefix-cached attention tokens/s; % HBM (decode) / % bf16 TC peak (extend)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 129 << 20           # GB300 L2
DEFAULT_WORKLOAD = "c5"
DEFAULT_SUBS = {"c5": ("c3", "c4", "c2", "c1")}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------- ncu traffic
# the sources of the attention call's kernels (the ones the recorded counters cover)
ATTENTION_SOURCES = ("attention_simt.cu", "decode_attention.cu", "extend_attention.cu", "rx_common.h",
                     "rx_device.cuh", "rx_kernels.h")


def kernel_source_hash() -> str:
    """Digest of the attention kernels' sources (CUDA files and the headers they include): DRAM
    counters recorded for one version of those kernels are reported only while it is unchanged."""
    import hashlib
    csrc = os.path.join(ROOT, "prefix_cached_kv_radix_gb300", "csrc")
    h = hashlib.sha256()
    for f in ATTENTION_SOURCES:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """dram__bytes_read.sum + dram__bytes_write.sum of the attention call's kernels for one
    step, from the committed ncu summary (profiles/traffic.json), or None when absent or
    taken on other kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    e = json.load(open(p)).get(workload)
    if not e or e.get("sources") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


# ---------------------------------------------------------------------------- work model
def algorithmic_work(w):
    """Attention FLOPs (4*D per causal (row, key) pair per q head) and unique bytes."""
    s = w.spec
    pairs = 0
    for b in range(w.batch):
        P, n = s.req_cached[b], s.req_new[b]
        pairs += n * P + n * (n + 1) // 2
    flops = 4.0 * s.d * s.hq * pairs
    elt = 4 if s.dtype == "f32" else 2
    row = s.hkv * s.d * elt * 2          # K + V per token
    # unique KV the step must read: union of the contexts (shared prefixes once)
    uniq = set()
    tot_ctx = 0
    for b in range(w.batch):
        path = w.seg_path(s.req_seg[b])
        c = s.req_cached[b]
        acc = 0
        for seg in path:
            take = min(s.seg_len[seg], c - acc)
            if take <= 0:
                break
            uniq.add((seg, take))
            acc += take
        tot_ctx += c + s.req_new[b]
    seg_take = {}
    for seg, take in uniq:
        seg_take[seg] = max(seg_take.get(seg, 0), take)
    uniq_tokens = sum(seg_take.values()) + w.total_new()
    qo_bytes = 2 * w.total_new() * s.hq * s.d * elt
    idx_bytes = 4 * tot_ctx
    return dict(flops=flops, pairs=pairs, kv_unique_bytes=uniq_tokens * row,
                bytes=uniq_tokens * row + qo_bytes + idx_bytes, kv_naive_bytes=tot_ctx * row,
                naive_bytes=tot_ctx * row + qo_bytes + idx_bytes)


def pool_write_bytes(w, stride: int) -> int:
    """kv_pool_write's algorithmic bytes: the new rows' K and V read and written once each, the
    slot table written in full ([batch, stride] int32), the prefix and new slot lists read."""
    s = w.spec
    elt = 4 if s.dtype == "f32" else 2
    T = w.total_new()
    return 4 * T * s.hkv * s.d * elt + 4 * w.batch * stride + 4 * (int(sum(s.req_cached)) + T)


# ---------------------------------------------------------------------------- clocks
# A separate process samples the clocks, so that the queries run on another core and never on
# the benchmark's own thread: an NVML query made by the benchmark's thread next to a short step
# (before it, after it, or during the L2 flush before it) was measured to add 7-15 us to a step.
_SAMPLER = r"""
import ctypes, os, sys, time
cores = os.sched_getaffinity(0)
if len(cores) > 1 and int(sys.argv[4]) in cores:   # off the core a step timed alone runs on
    os.sched_setaffinity(0, cores - {int(sys.argv[4])})
lib = ctypes.CDLL("libnvidia-ml.so.1")
assert lib.nvmlInit_v2() == 0
h = ctypes.c_void_p()
bus = sys.argv[1].encode()
if not bus or lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
    n = ctypes.c_uint()
    lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
    idx = 0 if n.value == 1 else int(sys.argv[2])
    assert lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) == 0
fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or lib.nvmlDeviceGetCurrentClocksThrottleReasons
period = float(sys.argv[3])
sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm))   # the first queries are the slow ones
lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
fn(h, ctypes.byref(rs))
print("ready", flush=True)
while True:   # the maximum clock is fixed: queried once above
    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and fn(h, ctypes.byref(rs)) == 0:
        print(sm.value, mx.value, rs.value, flush=True)
    time.sleep(period)
"""


class ClockSampler:
    """SM clock and throttle reasons of this process's GPU (read only), sampled every
    0.2 ms (plus the query's own time) by a separate process through NVML while the timed regions run (start/pause
    around each region); falls back to `nvidia-smi -lms 200` when NVML cannot be used."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.0002, avoid_core: int = -1):
        self.period = period_s
        self.dev = device_index
        self.avoid = avoid_core
        self.samples = []             # (sm_mhz, max_mhz, reasons bitmask)
        self.proc = None
        self.thread = None
        self.smi = False
        self.smi_lines = []
        self.bus = ""
        try:
            import torch
            pr = torch.cuda.get_device_properties(device_index)
            self.bus = f"{getattr(pr, 'pci_domain_id', 0):08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        except Exception:
            self.bus = ""

    def _reader(self, proc, sink):
        for ln in proc.stdout:
            sink.append(ln.strip())

    def start(self):
        """Start sampling (a no-op while sampling)."""
        if self.proc is not None:
            return
        lines = []
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", _SAMPLER, self.bus, str(self.dev), str(self.period),
                                          str(self.avoid)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline().strip()
            if first != "ready":
                raise OSError("sampler did not start")
            self.smi = False
        except (OSError, ValueError):
            if self.proc is not None:
                self.proc.kill()
            try:
                q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                     "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
                self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.bus or self.dev}", f"--query-gpu={q}",
                                              "--format=csv,noheader,nounits", "-lms", "200"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.smi = True
            except OSError:
                self.proc = None
                return
        self.thread = threading.Thread(target=self._reader, args=(self.proc, lines), daemon=True)
        self.thread.start()
        self._lines = lines

    def pause(self):
        """Stop sampling and keep what was sampled."""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        for ln in self._lines:
            f = ln.replace(",", " ").split()
            try:
                if self.smi:
                    if len(f) < 9:
                        continue
                    bits = 0
                    for name, val in zip((0x8, 0x40, 0x20, 0x4), f[5:9]):
                        if val.lower() in ("active", "1", "yes"):
                            bits |= name
                    self.samples.append((float(f[1]), float(f[2]), bits))
                else:
                    self.samples.append((float(f[0]), float(f[1]), int(f[2])))
            except (ValueError, IndexError):
                continue
        self.proc = None

    def stop(self):
        """Stop sampling; returns {sm_mhz (median), sm_max_mhz, sm_min_mhz, reasons, samples, source} or None."""
        self.pause()
        if not self.samples:
            return None
        smp = self.samples
        reasons = sorted({name for _, _, r in smp for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(x[0] for x in smp), "sm_max_mhz": max(x[1] for x in smp),
                "sm_min_mhz": min(x[0] for x in smp), "reasons": reasons, "samples": len(smp),
                "source": ("nvidia-smi every 200 ms during the timed regions" if self.smi else
                           f"NVML from a separate process, one query per {self.period * 1e3:.1f} ms sleep, during the timed regions")}


# ---------------------------------------------------------------------------- replicas
def reduce_max(values, world: int, device="cpu"):
    """Elementwise max over ranks (the timed region's slowest replica); identity at N = 1."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_throughput(tokens_per_step: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: every replica processes the same batch each step (weak scaling)."""
    return tokens_per_step * steps * world / (ms_max * 1e-3)


# ---------------------------------------------------------------------------- our arm
def fresh_prompts(w, step, used):
    """The workload's prompts with step-specific new-token ids.  Requests that diverge from
    the cache at the same point get distinct first tokens, which also differ from the
    cached continuation there and from every first token used there in earlier steps, so
    each step inserts exactly its new tokens as fresh leaves."""
    s = w.spec
    rng = np.random.default_rng([s.seed, 9000, step])
    prompts = []
    for b in range(w.batch):
        n = s.req_new[b]
        new = rng.integers(0, s.vocab, size=n).astype(np.int32)
        base = w.request_prefix_tokens(b)
        key = (s.req_seg[b], s.req_cached[b])
        if key not in used:
            forb = used[key] = set()
            path = w.path_tokens(s.req_seg[b])
            if s.req_cached[b] < len(path):
                forb.add(int(path[s.req_cached[b]]))
            for bb in range(w.batch):        # the workload's own first tokens at this point
                if (s.req_seg[bb], s.req_cached[bb]) == key and s.req_new[bb]:
                    forb.add(int(w.req_tokens[bb][0]))
        forb = used[key]
        if n:
            while int(new[0]) in forb:
                new[0] = int(rng.integers(0, s.vocab))
            forb.add(int(new[0]))
        prompts.append(np.concatenate([base, new]).astype(np.int32))
    return prompts


def link_rates(pairs, reps: int = 5):
    """Attainable host-link rates on this machine: one large cudaMemcpyAsync per direction from/to
    the same pinned buffers the e2e steps use (H2D alone, D2H alone, both at once on two
    streams), timed with CUDA events; GB/s (1e9 B/s), best of `reps`."""
    import torch
    h2d_src, h2d_dst, d2h_src, d2h_dst = pairs
    nb_in = h2d_src.numel() * h2d_src.element_size()
    nb_out = d2h_src.numel() * d2h_src.element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, streams):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in streams]
            for (a, _), st in zip(ev, streams):
                a.record(st)
            fn()
            for (_, b), st in zip(ev, streams):
                b.record(st)
            torch.cuda.synchronize()
            best = min(best, max(a.elapsed_time(b) for a, b in ev))
        return best

    def h2d():
        with torch.cuda.stream(s_in):
            h2d_dst.copy_(h2d_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            d2h_dst.copy_(d2h_src, non_blocking=True)

    t_in = timed(h2d, [s_in])
    t_out = timed(d2h, [s_out])
    t_both = timed(lambda: (h2d(), d2h()), [s_in, s_out])
    return {"h2d_gbs": nb_in / (t_in * 1e-3) / 1e9, "d2h_gbs": nb_out / (t_out * 1e-3) / 1e9,
            "both_gbs": (nb_in + nb_out) / (t_both * 1e-3) / 1e9, "h2d_bytes": nb_in, "d2h_bytes": nb_out,
            "how": "one cudaMemcpyAsync per direction between the e2e steps' pinned host buffers and device "
                   "rows, best of 5, CUDA events"}


def measure(name, args, rank, world, local_rank, cpu: bool):
    """Every figure of one workload: the step (value), the e2e step through host buffers, the
    attention call and kv_pool_write alone (rooflines), clocks, host link, CPU baseline."""
    import torch
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine, _dev_from_host

    dev = torch.device("cuda", local_rank)
    spec = W.config(name)
    if args.requests:
        spec = W.take_requests(spec, args.requests)
    if args.pool_slots:
        spec.num_slots = args.pool_slots
    w = W.generate(spec)
    s = spec
    eng = PrefixCacheEngine(s.dtype, s.hq, s.hkv, s.d, s.num_slots, s.seed, device=str(dev), poison=False)
    for i in range(len(s.histories)):
        k, v = w.history_kv(i)
        eng.populate(w.history_tokens(i), k, v)
    q, kn, vn = w.stacked_new()
    qd, kd, vd = (_dev_from_host(x, s.dtype, dev) for x in (q, kn, vn))
    out = torch.empty_like(qd)
    lse = torch.empty(qd.shape[0], s.hq, dtype=torch.float32, device=dev)
    # pinned host copies for the end-to-end variant, and a second set of device rows for it: the
    # steps use the two in turn, so a step's input copies run under the previous step's kernels
    qh, kh, vh = (x.cpu().pin_memory() for x in (qd, kd, vd))
    rows_e2e = [(qd, kd, vd), tuple(torch.empty_like(x) for x in (qd, kd, vd))]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    T = w.total_new()
    used = {}
    stream = torch.cuda.current_stream()
    att_ev, write_ev = [], []
    launches = [0]
    strides = []

    # every step's prompts are prepared before timing (inputs resident when timing starts)
    n_total = 2 * args.warmup + 4 * args.steps     # warm-up (both paths), value, e2e, attention, isolated
    step_inputs = []
    for i in range(n_total):
        prompts = fresh_prompts(w, i, used)
        ind = np.concatenate([[0], np.cumsum([len(x) for x in prompts])]).astype(np.int64)
        step_inputs.append((np.concatenate(prompts).astype(np.int32), ind))
    n_new = np.asarray(s.req_new, np.int32)   # the library's own type: no conversion per step
    group_mode = True if s.decode else "auto"

    def n_launch(grouped: bool, e2e: bool, stage_bytes: int) -> int:
        # kv_pool_write (plus the index-array copy kernel for host-buffer steps; device-row
        # steps copy arrays of at most 1 MiB inside kv_pool_write's launch and larger ones by
        # the copy engine), then for decode: (group map, shared chunks) + private chunks +
        # merge; for extend: extend, or (prep, shared tcgen05, private + merge) with groups
        base = 2 if e2e else 1
        if s.decode:
            return base + (2 if grouped else 0) + 2
        return base + (1 if not grouped else 3)

    def step(i, e2e=False):
        """One step through the library's one-call path (plan, then copy + kernels + finish);
        e2e: the new rows come from and the output goes to pinned host memory, through the
        library's own copies."""
        toks, ind = step_inputs[i]
        q_, k_, v_ = rows_e2e[i % 2] if e2e else (qd, kd, vd)
        plan = eng.step(toks, ind, n_new, q_, k_, v_, out, lse, decode=s.decode, groups=group_mode, evict_tokens=T,
                        host=(qh, kh, vh, out_h) if e2e else None, chunks=args.chunks, overlap=True)
        launches[0] += n_launch(plan.layout.num_groups > 0, e2e, int(plan.layout.bytes))
        return plan

    def step_att(i):
        """The same step through the per-operation calls, with CUDA events around kv_pool_write
        alone and around the attention call alone (the rooflines' kernel times)."""
        toks, ind = step_inputs[i]
        plan = eng.plan_concat(toks, ind, n_new, groups=group_mode)
        strides.append(plan.stride)
        d = eng.upload(plan)
        grp = eng.groups(plan, d)
        if hasattr(torch.cuda, "_sleep"):
            # keep the GPU busy while the host records the start event and issues the calls, so
            # that only the kernels fall between the events
            torch.cuda._sleep(200_000)
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        eng.write(plan, d, kd, vd)
        w1.record(stream)
        e0.record(stream)
        if s.decode:
            eng.decode(plan, d, qd, out, lse, groups=grp)
        else:
            eng.extend(plan, d, qd, out, lse)
        e1.record(stream)
        write_ev.append((w0, w1))
        att_ev.append((e0, e1))
        eng.finish(plan, evict_tokens=T)

    for i in range(args.warmup):
        step(i)
    for i in range(args.warmup):                # the host-buffer path's first use (copy streams, events)
        step(args.warmup + 3 * args.steps + i, e2e=True)
    torch.cuda.synchronize()
    if eng.device_status() != 0:
        raise RuntimeError(f"device status {eng.device_status()} after warm-up")

    work = algorithmic_work(w)
    # A step that touches far more than L2 holds is timed as K steps back to back in one event
    # region (the host's plan of step i+1 overlaps the GPU's step i, as the engine is built to
    # do: double-buffered staging, host finish right after the launch).  A step that fits in
    # L2 is timed alone after an L2 flush and a synchronize.
    back_to_back = work["bytes"] >= 2 * L2_BYTES
    cores = sorted(os.sched_getaffinity(0))
    pin_core = cores[-1 - local_rank % len(cores)]   # a core per rank, from the top
    clocks = ClockSampler(local_rank, avoid_core=pin_core)

    def timed(e2e, isolated=not back_to_back, first=None):
        # a step timed alone is host-bound: its thread stays on one core for the region (the
        # clock sampler keeps off that core), instead of resuming on another one, cold, after
        # each synchronize
        allowed = os.sched_getaffinity(0)
        if isolated and len(allowed) > 1:
            os.sched_setaffinity(0, {pin_core})
        try:
            return timed_region(e2e, isolated, first)
        finally:
            os.sched_setaffinity(0, allowed)

    def timed_region(e2e, isolated, first):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        launches[0] = 0
        first = args.warmup + (args.steps if e2e else 0) if first is None else first
        if not isolated:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)                  # created before timing starts (see below)
            e1.record(stream)
            torch.cuda.synchronize()
            clocks.start()
            e0.record(stream)
            for i in range(args.steps):
                step(first + i, e2e=e2e)
            e1.record(stream)
            torch.cuda.synchronize()
            clocks.pause()
            if world > 1:
                torch.distributed.barrier()
            return e0.elapsed_time(e1), launches[0]
        # the events exist before timing starts (an event's first record creates it, which would
        # otherwise fall inside the timed region)
        times = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for e0, e1 in times:
            e0.record(stream)
            e1.record(stream)
        clocks.start()
        for i in range(args.steps):
            flush.zero_()                      # untimed: evict L2 between timed steps
            # the flush completes before the timed region opens, so the step's host work
            # (planning, launches, finish) cannot hide behind it: the region holds the whole step
            torch.cuda.synchronize()
            e0, e1 = times[i]
            e0.record(stream)
            step(first + i, e2e=e2e)
            e1.record(stream)
        torch.cuda.synchronize()
        clocks.pause()
        if world > 1:
            torch.distributed.barrier()
        ms = sum(a.elapsed_time(b) for a, b in times)
        return ms, launches[0]

    ms, n_launches = timed(False)
    ms_e2e, _ = timed(True)
    clk = clocks.stop()
    ms_iso = None
    if back_to_back:   # the same steps once more, each alone after a flush, for comparison
        ms_iso, _ = timed(False, isolated=True, first=args.warmup + 3 * args.steps + args.warmup)
    for i in range(args.steps):                # kernel-only timing for the rooflines (untimed above)
        flush.zero_()                          # no synchronize: the host prepares the calls while the
        step_att(args.warmup + 2 * args.steps + i)   # flush runs, so only the kernels fall between the events
    torch.cuda.synchronize()
    if eng.device_status() != 0:
        raise RuntimeError(f"device status {eng.device_status()} after timed steps")
    link = link_rates((qh, rows_e2e[1][0], out, out_h))
    ms, ms_e2e = reduce_max([ms, ms_e2e], world, dev)
    hbm, bf16, bf16_s, src = load_peaks()
    att = statistics.median(a.elapsed_time(b) for a, b in att_ev)
    wr = statistics.median(a.elapsed_time(b) for a, b in write_ev)
    # the bound follows the step's arithmetic intensity against the ridge of the two peaks
    intensity = work["flops"] / work["bytes"]
    ridge = bf16 * 1e12 / (hbm * 1e9)
    traffic = recorded_traffic(s.name)
    if s.decode or s.dtype == "f32" or intensity < ridge:
        achieved = work["bytes"] / (att * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic,
                "kernel": "decode_attention (split-KV + merge)" if s.decode else "prefix_extend_attention",
                "algorithmic": f"{work['bytes'] / 1e9:.4f} GB unique (KV {work['kv_unique_bytes'] / 1e9:.4f} GB + Q/O + indices) per launch",
                "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                "launch_ms": att, "peak_source": f"{src} hbm_gbs (copy)"}
        if s.decode:
            naive = work["naive_bytes"] / (att * 1e-3) / 1e9
            roof["naive"] = {"achieved": naive, "frac": naive / hbm,
                             "algorithmic": f"{work['naive_bytes'] / 1e9:.4f} GB: every request's whole context "
                                            "read as if nothing were shared (labelled, not the headline fraction)"}
    else:
        # the attention call is timed alone (after an L2 flush, with nothing else running): the
        # burst peak applies; the fraction of the sustained peak is given beside it
        achieved = work["flops"] / (att * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s", "frac": achieved / bf16,
                "traffic": traffic, "kernel": "prefix_extend_attention (tcgen05)",
                "algorithmic": f"{work['flops'] / 1e9:.3f} GFLOP per launch (4*D per causal pair per q head)",
                "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                "launch_ms": att, "peak_source": f"{src} bf16_tflops (burst: the kernel is timed alone)",
                "frac_of_sustained": achieved / bf16_s if bf16_s else None}
    roof["traffic_note"] = ("dram read+write bytes of the attention call's kernels for one step (ncu, "
                            "profiles/traffic.json)" if traffic is not None else
                            "null: no ncu capture recorded for these kernel sources")
    wbytes = pool_write_bytes(w, int(statistics.median(strides)))
    wach = wbytes / (wr * 1e-3) / 1e9
    pool_roof = {"bound": "hbm", "achieved": wach, "peak": hbm, "unit": "GB/s", "frac": wach / hbm, "launch_ms": wr,
                 "algorithmic": f"{wbytes / 1e6:.2f} MB per launch (new K/V read + written, slot table, slot lists)"}
    value = replica_throughput(T, args.steps, world, ms)
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = out_h.numel() * out_h.element_size()
    e2e_copy = (h2d + d2h) / (ms_e2e / args.steps * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if s.dtype == "f32" else "bf16", "data": "synthetic (seeded N(0,1) Q/K/V, uniform token ids)",
        "config": {"workload": f"{s.name}: {s.note}", "batch": w.batch, "new_tokens_per_step": T,
                   "cached_prefix_tokens": int(sum(s.req_cached)), "heads": f"{s.hq}/{s.hkv}x{s.d}",
                   "kv_pool_slots": s.num_slots,
                   "l2": (f"not flushed: a step touches {work['bytes'] / 1e9:.2f} GB (L2 {L2_BYTES >> 20} MiB); "
                          f"{args.steps} steps back to back in one timed region" if back_to_back else
                          f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write), each step timed alone"),
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "kv_pool_write_roofline": pool_roof,
        "cpu_baseline": cpu_baseline(w, args.cpu_seconds) if (cpu and rank == 0) else None,
        "e2e": {"value": replica_throughput(T, args.steps, world, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "copy_gbs": e2e_copy,
                "frac_of_link": e2e_copy / link["both_gbs"] if link["both_gbs"] else None},
        "host_link": link,
        "gpu_launches": n_launches,   # library kernels in the timed region (value); the e2e region adds one per step
        "isolated_step_ms": ms_iso / args.steps if ms_iso is not None else None,
        "clocks": clk,
        "radix_stats": eng.tree.stats(),
    }
    return line


def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    import gc

    def one(name):
        r = measure(name, args, rank, world, local_rank, cpu=not args.no_cpu_baseline)
        gc.collect()                   # the workload's pools and rows go before the next one's
        torch.cuda.empty_cache()
        return r

    line = one(args.workload)
    subs = {}
    for name in args.subs:
        if name != args.workload:
            subs[name] = one(name)
            for k in ("metric", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline",
                      "data"):
                subs[name].pop(k, None)
    if subs:
        line["sub_results"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- oracle timing
def _f32(a, dtype):
    return W.bf16_bits_to_f32(a) if dtype == "bf16" else np.asarray(a, np.float32)


def oracle_step(w, rows_of=None, threads: int = 0, full: bool = False):
    """The oracle's own version of one step: list matcher + slot allocator replay for the
    table, fp64 attention for the output rows.  rows_of(b) gives the row indices of request b
    to compute (None: every new row); full=True computes every row of the whole prompt, as an
    uncached recompute must.  Returns (new tokens output, threads, keys attended per head,
    seconds in the matcher)."""
    import oracle
    s = w.spec
    lm = oracle.ListMatcher()
    for i in range(len(s.histories)):
        lm.add(w.history_tokens(i), np.zeros(len(w.history_tokens(i)), np.int32))
    done, keys, t_match = 0, 0, 0.0
    for b in range(w.batch):
        t0 = time.perf_counter()
        lm.match(w.request_tokens(b))
        t_match += time.perf_counter() - t0
        n, P = s.req_new[b], s.req_cached[b]
        idx = np.arange(n) if rows_of is None else np.asarray(rows_of(b), np.int64)
        if len(idx) == 0 and not full:
            continue
        k, v = w.request_kv(b)
        k, v = _f32(k, s.dtype), _f32(v, s.dtype)
        q = _f32(w.req_q[b], s.dtype)
        if full:
            # no cache: every position of the prompt is computed (the prefix rows' queries are
            # seeded draws of the same distribution; only the work matters here)
            qp = np.random.default_rng([s.seed, 77, b]).standard_normal((P, s.hq, s.d), dtype=np.float32)
            qa = np.concatenate([_f32(W.f32_to_bf16_bits(qp), "bf16") if s.dtype == "bf16" else qp, q])
            pos = np.arange(P + n)
            oracle.attention_rows(qa, pos, k, v, s.scale, threads)
            keys += int((pos + 1).sum())
        else:
            oracle.attention_rows(q[idx], P + idx, k, v, s.scale, threads)
            keys += int((P + idx + 1).sum())
        done += len(idx)
    return done, (threads or oracle.max_threads()), keys, t_match


# Rows per request in one baseline step where a full step would take minutes: c5's 32
# requests x 1024 rows over ~30 K keys (32 TFLOP) are sampled.  The reference arm, which runs
# --steps oracle steps, also samples c3 (its full step takes tens of seconds on the host).
def sample_rows(name, reference: bool = False):
    if name.startswith("c5"):
        return lambda b: np.array([0, 1023])
    if reference and name.startswith("c3"):
        return lambda b: np.arange(8)
    return None


def sample_note(name, reference: bool = False):
    if name.startswith("c5"):
        return "new rows {0, 1023} of every request"
    if reference and name.startswith("c3"):
        return "the first 8 new rows of every request"
    return None


def _timed_loop(fn, seconds, min_reps=1):
    t0 = time.perf_counter()
    reps, acc = 0, []
    while True:
        acc.append(fn())
        reps += 1
        if reps >= min_reps and time.perf_counter() - t0 > seconds:
            break
    return time.perf_counter() - t0, reps, acc


def cpu_baseline(w, seconds):
    """Time the oracle (as it stands) on the host cores on a bounded sample of the step: the rows
    mode on all cores (the headline baseline), plus for the small workloads a 1-core run and the
    uncached full recompute, the list matcher alone, and for the sampled workload the full step
    extrapolated from the sample (labelled as such)."""
    import oracle
    oracle.build()
    s = w.spec
    rows_of = sample_rows(s.name)
    dt, reps, acc = _timed_loop(lambda: oracle_step(w, rows_of), seconds)
    toks = sum(a[0] for a in acc)
    thr = acc[0][1]
    sample = (f"{reps} full oracle step(s) of {s.name} (list matcher + fp64 attention of every new row)"
              if rows_of is None else
              f"{reps} oracle pass(es) of {s.name} with {sample_note(s.name)}")
    res = {"value": toks / dt, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample, "seconds": dt,
           "mode": "rows (the rows the method outputs, over logical-order K/V)"}
    # the list matcher alone: one step's prompts against the cached sequences
    t_match = sum(a[3] for a in acc) / reps
    ptoks = sum(len(w.request_tokens(b)) for b in range(w.batch))
    res["matcher"] = {"seconds_per_step": t_match, "prompt_tokens_per_s": ptoks / t_match if t_match else None,
                      "what": "oracle list matcher (longest common prefix over the cached sequences), one step"}
    if rows_of is not None:
        keys_s = sum(a[2] for a in acc)
        t_att = dt - t_match * reps
        keys_full = sum(s.req_new[b] * (s.req_cached[b] + 1) + s.req_new[b] * (s.req_new[b] - 1) // 2
                        for b in range(w.batch))
        est = t_att / keys_s * keys_full + t_match
        res["extrapolated_full_step"] = {
            "label": "EXTRAPOLATION, not a measurement: the sampled rows' time per attended key scaled to every new "
                     "row of the step, plus the matcher",
            "seconds_per_step": est, "value": w.total_new() / est, "unit": UNIT}
    if s.name in ("c1", "c2"):
        d1, r1, a1 = _timed_loop(lambda: oracle_step(w, rows_of, threads=1), seconds / 2)
        res["one_core"] = {"value": sum(a[0] for a in a1) / d1, "unit": UNIT, "cores": 1, "seconds": d1,
                           "sample": f"{r1} full oracle step(s) on one thread"}
        df, rf, af = _timed_loop(lambda: oracle_step(w, full=True), seconds / 2)
        res["full_mode"] = {"value": sum(a[0] for a in af) / df, "unit": UNIT, "cores": thr, "seconds": df,
                            "rows_per_step": int(sum(s.req_cached) + w.total_new()),
                            "sample": f"{rf} uncached step(s): every row of every prompt recomputed; value counts "
                                      "the new tokens delivered"}
    return res


def run_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec = W.config(args.workload)
    w = W.generate(spec)
    rows_of = sample_rows(spec.name, reference=True)
    note = sample_note(spec.name, reference=True)
    for _ in range(args.warmup):
        oracle_step(w, rows_of)
    t0 = time.perf_counter()
    toks = 0
    thr = 1
    for _ in range(args.steps):
        n, thr, _, _ = oracle_step(w, rows_of)
        toks += n
    dt = time.perf_counter() - t0
    v = toks / dt
    sample = (f"{args.steps} oracle steps of {spec.name} (list matcher + fp64 attention of every new row)"
              if rows_of is None else
              f"{args.steps} oracle steps of {spec.name}, each {note}")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": f"{spec.name}: {spec.note}", "batch": w.batch,
                       "sample": "full step" if rows_of is None else note},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.CONFIG_NAMES))
    ap.add_argument("--subs", default=None,
                    help="comma-separated workloads measured in the same run (default: c3,c4,c2,c1 with c5; "
                         "none otherwise); 'none' for none")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunks", type=int, default=0,
                    help="request ranges of the e2e copy pipeline (0: chosen by the library)")
    ap.add_argument("--requests", type=int, default=0,
                    help="profiling only: the workload's first N requests (same per-request shapes)")
    ap.add_argument("--pool-slots", type=int, default=0,
                    help="override the KV pool size (profiling captures keep the device footprint small)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.subs is None:
        args.subs = list(DEFAULT_SUBS.get(args.workload, ()))
    elif args.subs in ("", "none"):
        args.subs = []
    else:
        args.subs = [x for x in args.subs.split(",") if x]
        for x in args.subs:
            if x not in W.CONFIG_NAMES:
                ap.error(f"unknown workload {x}")
    if args.requests or args.pool_slots:
        args.subs = []                  # profiling captures: one workload
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
