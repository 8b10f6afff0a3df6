"""Benchmark: prefix-cached attention steps on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload c2]

One step is one pass of the whole hot path over one batch: host radix match and slot
allocation, upload of the step's index arrays, kv_pool_write (slot table + K/V scatter),
the attention kernel(s) (extend, or split-KV decode + merge), insert of the new tokens
and LRU eviction of as many cached tokens (so the cache stays at a steady size).  Every
step's requests carry fresh new-token ids, so each step is a new batch of requests that
hits the cached prefix.  Inputs (Q and the new K/V) are resident in HBM when the timed
region starts; the e2e figure repeats the step through the same public call with the inputs
in pinned host memory: the library copies them in and the output back inside the timed
region (a pipeline of request ranges whose copies run behind the kernels).

Prints one JSON line.  With N > 1 (torchrun) every rank runs its own replica of the
workload on its own GPU (the path shards over independent requests; no collective is
needed), value = all ranks' tokens / max over ranks of the time.
"""
from __future__ import annotations

import argparse
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
                bytes=uniq_tokens * row + qo_bytes + idx_bytes, kv_naive_bytes=tot_ctx * row)


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names[1:], f[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


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


def run_ours(args, rank, world, local_rank):
    import torch
    from prefix_cached_kv_radix_gb300.engine import PrefixCacheEngine, _dev_from_host

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    spec = W.config(args.workload)
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
    att_ev = []
    launches = [0]

    # every step's prompts are prepared before timing (inputs resident when timing starts)
    n_total = 2 * args.warmup + 4 * args.steps     # warm-up (both paths), value, e2e, attention, isolated
    step_inputs = []
    for i in range(n_total):
        prompts = fresh_prompts(w, i, used)
        ind = np.concatenate([[0], np.cumsum([len(x) for x in prompts])]).astype(np.int64)
        step_inputs.append((np.concatenate(prompts).astype(np.int32), ind))
    n_new = np.asarray(s.req_new, np.int64)
    group_mode = True if s.decode else "auto"

    def n_launch(grouped: bool, e2e: bool, stage_bytes: int) -> int:
        # kv_pool_write (plus the index-array copy kernel for host-buffer steps and for index
        # arrays of at most 1 MiB; larger ones of device-row steps go by the copy engine), then
        # for decode: (group map, shared chunks) + private chunks + merge; for extend: extend,
        # or (prep, shared tcgen05, private + merge) with groups
        base = 2 if (e2e or stage_bytes <= (1 << 20)) else 1
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
        """The same step through the per-operation calls, with CUDA events around the attention
        call alone (the roofline's kernel time)."""
        toks, ind = step_inputs[i]
        plan = eng.plan_concat(toks, ind, n_new, groups=group_mode)
        d = eng.upload(plan)
        grp = eng.groups(plan, d)
        eng.write(plan, d, kd, vd)
        if hasattr(torch.cuda, "_sleep"):
            # keep the GPU busy while the host records the start event and issues the call, so
            # that only the attention kernels fall between the events
            torch.cuda._sleep(100_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if s.decode:
            eng.decode(plan, d, qd, out, lse, groups=grp)
        else:
            eng.extend(plan, d, qd, out, lse)
        e1.record(stream)
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

    def timed(e2e, isolated=not back_to_back, first=None):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        launches[0] = 0
        first = args.warmup + (args.steps if e2e else 0) if first is None else first
        if not isolated:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(args.steps):
                step(first + i, e2e=e2e)
            e1.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            return e0.elapsed_time(e1), launches[0]
        times = []
        for i in range(args.steps):
            flush.zero_()                      # untimed: evict L2 between timed steps
            # the flush completes before the timed region opens, so the step's host work
            # (planning, launches, finish) cannot hide behind it: the region holds the whole step
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(first + i, e2e=e2e)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ms = sum(a.elapsed_time(b) for a, b in times)
        return ms, launches[0]

    clocks = ClockSampler(local_rank)
    clocks.start()
    ms, n_launches = timed(False)
    ms_e2e, _ = timed(True)
    clk = clocks.stop()
    ms_iso = None
    if back_to_back:   # the same steps once more, each alone after a flush, for comparison
        ms_iso, _ = timed(False, isolated=True, first=args.warmup + 3 * args.steps + args.warmup)
    for i in range(args.steps):                # attention-only timing for the roofline (untimed above)
        flush.zero_()                          # no synchronize: the host prepares the call while the
        step_att(args.warmup + 2 * args.steps + i)   # flush runs, so only the kernels fall between the events
    torch.cuda.synchronize()
    if eng.device_status() != 0:
        raise RuntimeError(f"device status {eng.device_status()} after timed steps")
    ms, ms_e2e = reduce_max([ms, ms_e2e], world, dev)
    att_ms = [a.elapsed_time(b) for a, b in att_ev]
    hbm, bf16, bf16_s, src = load_peaks()
    att = statistics.median(att_ms) if att_ms else float("nan")
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
                "launch_ms": att, "peak_source": f"{src} hbm_gbs"}
    else:
        achieved = work["flops"] / (att * 1e-3) / 1e12
        # a kernel timed inside long steps runs under the power cap: the sustained peak applies
        long_steps = ms / args.steps >= 5.0
        peak = bf16_s if long_steps and bf16_s else bf16
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic, "kernel": "prefix_extend_attention (tcgen05)",
                "algorithmic": f"{work['flops'] / 1e9:.3f} GFLOP per launch (4*D per causal pair per q head)",
                "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                "launch_ms": att,
                "peak_source": f"{src} " + ("bf16_tflops_sustained (steps of >= 5 ms)" if peak == bf16_s and long_steps
                                            else "bf16_tflops (burst)")}
    roof["traffic_note"] = ("dram read+write bytes of the attention call's kernels for one step (ncu, "
                            "profiles/traffic.json)" if traffic is not None else
                            "null: no ncu capture recorded for these kernel sources")
    tokens = T * args.steps * world
    value = replica_throughput(T, args.steps, world, ms)
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = out_h.numel() * out_h.element_size()
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
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
        "cpu_baseline": cpu,
        "e2e": {"value": replica_throughput(T, args.steps, world, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": n_launches,   # library kernels in the timed region (value); the e2e region adds one per step
        "isolated_step_ms": ms_iso / args.steps if ms_iso is not None else None,
        "clocks": clk,
        "radix_stats": eng.tree.stats(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- oracle timing
def oracle_step(w, rows_per_request=None):
    """The oracle's own version of one step: list matcher + slot allocator replay for the
    table, fp64 attention for the output rows.  Returns (tokens computed, threads)."""
    import oracle
    s = w.spec
    lm = oracle.ListMatcher()
    for i in range(len(s.histories)):
        lm.add(w.history_tokens(i), np.zeros(len(w.history_tokens(i)), np.int32))
    done = 0
    for b in range(w.batch):
        lm.match(w.request_tokens(b))
        n = s.req_new[b]
        idx = np.arange(n) if rows_per_request is None else np.arange(min(n, rows_per_request))
        if len(idx) == 0:
            continue
        k, v = w.request_kv(b)
        k = W.bf16_bits_to_f32(k) if s.dtype == "bf16" else k
        v = W.bf16_bits_to_f32(v) if s.dtype == "bf16" else v
        q = W.bf16_bits_to_f32(w.req_q[b]) if s.dtype == "bf16" else w.req_q[b]
        oracle.attention_rows(q[idx], s.req_cached[b] + idx, k, v, s.scale)
        done += len(idx)
    return done, oracle.max_threads()


# Rows per request in one reference step (None = every new row): full steps where the oracle
# finishes one in about a second or two, a bounded sample of each request's rows otherwise.
REF_ROWS = {"c3": 8, "c5": 2}


def cpu_baseline(w, seconds):
    """Time the oracle (as it stands) on the host cores on a bounded sample of the step."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    toks, reps = 0, 0
    rows = None
    s = w.spec
    if s.name in REF_ROWS:
        rows = REF_ROWS[s.name]   # a few rows per request: full rows would take minutes to hours
    while True:
        n, thr = oracle_step(w, rows)
        toks += n
        reps += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    sample = (f"{reps} full oracle step(s) of {s.name} (list matcher + fp64 attention of every new row)"
              if rows is None else f"{reps} oracle pass(es) of {s.name} with the first {rows} new rows per request")
    return {"value": toks / dt, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample, "seconds": dt}


def run_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec = W.config(args.workload)
    w = W.generate(spec)
    rows = REF_ROWS.get(spec.name)
    for _ in range(args.warmup):
        oracle_step(w, rows)
    t0 = time.perf_counter()
    toks = 0
    thr = 1
    for _ in range(args.steps):
        n, thr = oracle_step(w, rows)
        toks += n
    dt = time.perf_counter() - t0
    v = toks / dt
    sample = (f"{args.steps} oracle steps of {spec.name} (list matcher + fp64 attention of every new row)"
              if rows is None else
              f"{args.steps} oracle steps of {spec.name}, each the first {rows} new rows of every request")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": f"{spec.name}: {spec.note}", "batch": w.batch,
                       "sample": "full step" if rows is None else f"first {rows} new rows per request"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2", choices=list(W.CONFIG_NAMES))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunks", type=int, default=0,
                    help="request ranges of the e2e copy pipeline (0: chosen by the library)")
    ap.add_argument("--requests", type=int, default=0,
                    help="profiling only: the workload's first N requests (same per-request shapes)")
    ap.add_argument("--pool-slots", type=int, default=0,
                    help="override the KV pool size (profiling captures keep the device footprint small)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
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
