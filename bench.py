"""Benchmark of paged decode attention on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one paged_attn_decode call (split kernel + log-sum-exp merge) over
one batch of the chosen seeded synthetic workload, inputs resident in HBM.
``value`` is whole-job KV throughput (algorithmic KV bytes of every rank's
step / max over ranks of the step time), in GB/s.  Between timed steps the L2
is not flushed; instead the KV bytes a step reads exceed the L2 (129 MB), by
rotating through several independent KV pools when one pool is smaller.
``--impl reference`` times the float64 CPU oracle on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention µs/step and KV GB/s (% of GB300 HBM peak), 1 GPU"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank's step time).  The
    replicas exchange nothing else: the path itself has no collective."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(step_bytes_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job KV throughput: every rank's step bytes over the slowest rank's step time."""
    return step_bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def cpu_oracle_steps(config: str, budgets, threads: int = 1, impl: str = "c"):
    """Time a float64 oracle on bounded samples of the workload, one sample per
    entry of ``budgets`` (seconds of oracle time; whole sequences are added until
    the budget is spent, at least one per sample), all in one child process.
    Sequences are taken in a fixed random order of the workload's length mix and
    each sample continues where the previous one stopped (cycling); a sequence's
    synthetic contents are generated once and reused.  impl "c": the plain-C
    oracle with ``threads`` OpenMP threads (0 = all host cores); impl "numpy": the
    NumPy oracle, single-threaded BLAS.  Returns (list of per-sample dicts with
    gbs / seqs / tokens / seconds, threads used, description)."""
    code = f"""
import json, os, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import oracle
from oracle import c_oracle
from paged_kv_decode_06_gb300 import workloads as wl
mla = {config!r} in wl.MLA_CONFIGS
spec = wl.MLA_CONFIGS[{config!r}] if mla else wl.CONFIGS[{config!r}]
rng = np.random.default_rng(spec.seed)
sl, ql, qsl, bt, pool = wl.draw_metadata(spec, rng)
order = np.random.default_rng(123).permutation(spec.num_seqs)
impl, threads = {impl!r}, {threads}
used = c_oracle.max_threads() if (impl == "c" and threads <= 0) else (threads if impl == "c" else 1)
cache, cached_bytes = {{}}, 0

def sequence(k):
    # the k-th sequence of the order, in a private pool holding only its pages
    # (same shapes and value distribution as the workload)
    global cached_bytes
    if k in cache:
        return cache[k]
    i = int(order[k % len(order)])
    L = int(sl[i]); q = int(ql[i]); n = (L + 15) // 16
    if mla:
        sub = wl.custom_mla_spec(num_q_heads=spec.num_q_heads, kv_dtype=spec.kv_dtype, seq_lens=(L,),
                                 query_len_choices=(q,), pool_pages=n, kv_scale=spec.kv_scale,
                                 fp8_source_scale=spec.fp8_source_scale, seed=k)
        w = wl.make_mla_workload(sub)
    else:
        sub = wl.custom_spec(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                             kv_dtype=spec.kv_dtype, seq_lens=(L,), query_len_choices=(q,), pool_pages=n,
                             k_scale=spec.k_scale, v_scale=spec.v_scale, fp8_source_scale=spec.fp8_source_scale,
                             seed=k, token_scale_range=spec.token_scale_range)
        w = wl.make_workload(sub)
    if cached_bytes + w.kv_bytes() <= (2 << 30):
        cache[k] = (w, L)
        cached_bytes += w.kv_bytes()
    return w, L

def run(w):
    if mla:
        c_oracle.run_mla_workload(w, threads=used) if impl == "c" else oracle.run_mla_workload(w)
    else:
        c_oracle.run_workload(w, threads=used) if impl == "c" else oracle.run_workload(w)

k = 0
out = []
for budget in {list(budgets)!r}:
    done_bytes = 0; t_used = 0.0; nseq = 0; ntok = 0
    while nseq == 0 or t_used < budget:
        w, L = sequence(k % len(order))
        t0 = time.perf_counter()
        run(w)
        t_used += time.perf_counter() - t0
        done_bytes += w.kv_bytes(); nseq += 1; ntok += L; k += 1
    out.append({{"gbs": done_bytes / t_used / 1e9, "seqs": nseq, "tokens": ntok, "seconds": t_used}})
print(json.dumps({{"steps": out, "threads": used}}))
"""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env.pop(k, None)
    if impl == "numpy":
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[k] = "1"
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=600 + 3 * sum(budgets))
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    what = (f"plain-C float64 oracle, {d['threads']} OpenMP thread(s)" if impl == "c"
            else "float64 NumPy oracle, single-threaded BLAS")
    return d["steps"], d["threads"], what


def cpu_oracle_sample(config: str, budget_s: float = 15.0, threads: int = 1, impl: str = "c"):
    """One bounded sample (``cpu_oracle_steps`` with one budget).  Returns (GB/s
    of KV processed, threads used, sample text)."""
    steps, used, what = cpu_oracle_steps(config, [budget_s], threads, impl)
    d = steps[0]
    sample = (f"{what}, {d['seqs']} whole sequences ({d['tokens']} cached tokens) drawn from the {config} "
              f"workload's length mix, {d['seconds']:.1f} s of oracle time")
    return d["gbs"], used, sample


def cpu_baseline(config: str, budget_s: float):
    """The ``cpu_baseline`` object: the C oracle on all host cores (value), on
    one core, and the NumPy oracle on one core, each on its own bounded sample
    (MLA workloads: the MLA oracles)."""
    gbs, cores, sample = cpu_oracle_sample(config, budget_s=0.4 * budget_s, threads=0, impl="c")
    g1, _, s1 = cpu_oracle_sample(config, budget_s=0.3 * budget_s, threads=1, impl="c")
    gn, _, sn = cpu_oracle_sample(config, budget_s=0.3 * budget_s, threads=1, impl="numpy")
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
            "host_cores": os.cpu_count(), "host_cpu": _cpu_model(),
            "single_core": {"value": g1, "unit": "GB/s", "cores": 1, "sample": s1},
            "numpy_single_core": {"value": gn, "unit": "GB/s", "cores": 1, "sample": sn}}


# Arm "CPU part" ids (/proc/cpuinfo) of the server cores an Arm host may have.
_ARM_PARTS = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2", "0xd4f": "Neoverse-V2",
              "0xd8e": "Neoverse-N3", "0xd84": "Neoverse-V3"}


def _cpu_model() -> str:
    """The host CPU's model name: lscpu's "Model name" (with its vendor),
    else /proc/cpuinfo's "model name", else the Arm part id mapped to its core
    name (Arm hosts list only the part id there); the part id is appended."""
    name, part = None, None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        fields = {}
        for line in r.stdout.splitlines():
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip(), v.strip())
        if fields.get("Model name", "-") != "-":
            vendor = fields.get("Vendor ID", "")
            name = fields["Model name"] if vendor in ("", "-") or vendor in fields["Model name"] else \
                f"{vendor} {fields['Model name']}"
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key == "model name" and name is None:
                    name = line.split(":", 1)[1].strip()
                elif key == "cpu part" and part is None:
                    part = line.split(":", 1)[1].strip().lower()
    except OSError:
        pass
    if name is None and part is not None:
        name = _ARM_PARTS.get(part, "Arm core")
    if name is None:
        import platform
        name = platform.machine()
    return f"{name} (CPU part {part})" if part else name


def _packed_views(parts, device):
    """One buffer holding several tensors back to back (each 16-byte aligned):
    returns (buffer, [views]).  parts = [(shape, dtype)]."""
    import torch
    offs, off = [], 0
    for shape, dtype in parts:
        n = int(math.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        offs.append((off, n))
        off += (n + 15) // 16 * 16
    if device == "pinned":
        buf = torch.empty(max(off, 16), dtype=torch.uint8).pin_memory()
    else:
        buf = torch.empty(max(off, 16), dtype=torch.uint8, device=device)
    views = [buf[o:o + n].view(dtype).view(shape) for (o, n), (shape, dtype) in zip(offs, parts)]
    return buf, views


def _timed_passes(step, ev_opts_for, pools, args, world, local, dev):
    """Warm-up, CUDA-graph capture and the timed passes of a decode benchmark.
    step(k, opts=None, stream_=None) enqueues step k (pool k % pools) on
    stream_ (None: the current stream); ev_opts_for(pidx, ev_a, ev_b) gives
    pool pidx's options with the split kernel's start / stop events.

    The decode step runs as an engine runs it: captured in CUDA graphs and
    replayed, so the device time is not hidden behind Python's per-call
    marshalling.  A graph holds GSTEP consecutive steps (rotating the KV pools),
    so the programmatic-dependent-launch overlap between steps survives inside
    it; single-step graphs cover a remainder.  Pass 1 (value): a timed window of
    exactly K steps back to back, bracketed by barrier + synchronize, repeated
    until the windows add up to at least --min-seconds (the same repeat count on
    every rank); ms per step = the median window.  Pass 2 (roofline): the split
    kernel's own duration, step by step, from external event records (at least
    200 steps).  Pass 3: K steps as direct calls through the binding (no graph).
    The clock sampler runs across passes 1 and 2.  Returns (ms per step, max
    over ranks; split-kernel ms list; direct ms; clocks; repeat count)."""
    import torch

    from paged_kv_decode_06_gb300 import binding
    stream = torch.cuda.current_stream()
    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    assert binding.paged_attn_device_status(clear=True) == 0
    cap = torch.cuda.Stream()
    gstep = pools * max(1, 8 // pools)

    def capture(first, n, opts=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for j in range(n):
                step(first + j, opts=opts, stream_=cap)
        return g

    big = capture(0, gstep)
    singles = [capture(pidx, 1) for pidx in range(pools)]

    def run_steps(count):
        k = 0
        while k + gstep <= count:
            big.replay()
            k += gstep
        while k < count:
            singles[k % pools].replay()
            k += 1
    ev_a = torch.cuda.Event(enable_timing=True)
    ev_b = torch.cuda.Event(enable_timing=True)
    ev_a.record(stream); ev_b.record(stream)     # torch times only events it has recorded once itself
    torch.cuda.synchronize()
    rgraphs = [capture(pidx, 1, opts=ev_opts_for(pidx, ev_a, ev_b)) for pidx in range(pools)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # graph warm-up, which also sizes the repeat count
    n_est = max(args.warmup, 4 * gstep)
    t_begin.record(stream)
    run_steps(n_est)
    t_end.record(stream)
    torch.cuda.synchronize()
    est_ms = t_begin.elapsed_time(t_end) / n_est
    repeats = max(1, math.ceil(args.min_seconds * 1e3 / max(1e-6, args.steps * est_ms)))
    repeats = int(max_over_ranks(float(min(repeats, 100000)), world, device=dev))
    windows = []
    with ClockSampler(local) as clk:
        for _ in range(repeats):
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            t_begin.record(stream)
            run_steps(args.steps)
            t_end.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            windows.append(t_begin.elapsed_time(t_end) / args.steps)
        split_ms = []
        for k in range(max(args.steps, 200)):
            rgraphs[k % pools].replay()
            ev_b.synchronize()
            split_ms.append(ev_a.elapsed_time(ev_b))
    ms = statistics.median(windows)
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for k in range(args.steps):
        step(k)
    d1.record(stream)
    torch.cuda.synchronize()
    direct_ms = d0.elapsed_time(d1) / args.steps
    return max_over_ranks(ms, world, device=dev), split_ms, direct_ms, clk.summary(), repeats


def _packed_e2e(base, works, out, lse, dev, prepare, args):
    """End to end through the public API: every step copies its inputs (q,
    block table, lengths, query starts) from pinned host memory and reads out /
    lse back; each direction is one copy of one packed buffer whose views are the
    tensors the call takes.  prepare(pool, q, bt, sl, qsl, out, lse) returns the
    binding's prepared call (arguments marshalled once, as a serving loop with
    static buffers holds it) of pool `pool` on those device views; step k runs
    pool k % pools's call.

    Two schedules, both with every step's copies inside the timed region:
    pipelined, as a serving loop runs them (the copy in of step k + 1 and the
    copy out of step k - 1 on their own streams while step k computes; device
    input and output buffers double-buffered, events order each buffer's
    reuse), and serial (copy in, call, copy out on one stream).  Afterwards a
    few pipelined steps, each followed by a synchronize, have their copied-back
    results compared bit for bit with the same call on the workload's own
    device tensors.  Returns (pipelined ms per step, serial ms per step, H2D
    bytes, D2H bytes, steps verified, all equal)."""
    import torch
    has_qsl = base.query_start_loc is not None
    in_parts = [(tuple(base.q.shape), base.q.dtype), (tuple(base.block_tables.shape), torch.int32),
                (tuple(base.seq_lens.shape), torch.int32)]
    if has_qsl:
        in_parts.append((tuple(base.query_start_loc.shape), torch.int32))
    out_parts = [(tuple(out.shape), out.dtype), (tuple(lse.shape), lse.dtype)]
    d_in, d_views, d_out, d_oviews, h_out, h_oviews = [], [], [], [], [], []
    for _ in range(2):
        b, v = _packed_views(in_parts, dev)
        d_in.append(b)
        d_views.append(v)
        b, v = _packed_views(out_parts, dev)
        d_out.append(b)
        d_oviews.append(v)
        b, v = _packed_views(out_parts, "pinned")
        h_out.append(b)
        h_oviews.append(v)
    h_ins = []
    for w in works:
        h_in, hv = _packed_views(in_parts, "pinned")
        hv[0].copy_(w.q.cpu())
        hv[1].copy_(torch.from_numpy(base.block_tables))
        hv[2].copy_(torch.from_numpy(base.seq_lens))
        if has_qsl:
            hv[3].copy_(torch.from_numpy(base.query_start_loc))
        h_ins.append(h_in)
    pools = len(works)

    calls = {}
    for pidx in range(pools):
        for x in range(2):
            v, ov = d_views[x], d_oviews[x]
            calls[(pidx, x)] = prepare(pidx, v[0], v[1], v[2], v[3] if has_qsl else None, ov[0], ov[1])

    def api_call(k, x):
        calls[(k % pools, x)]()

    comp = torch.cuda.current_stream()
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]

    def pipelined_step(k):
        x = k & 1
        if k >= 2:
            s_in.wait_event(in_free[x])      # step k - 2's call has read this input buffer
        with torch.cuda.stream(s_in):
            d_in[x].copy_(h_ins[k % pools], non_blocking=True)
        in_ready[x].record(s_in)
        comp.wait_event(in_ready[x])
        if k >= 2:
            comp.wait_event(out_free[x])     # step k - 2's results have been copied out
        api_call(k, x)
        in_free[x].record(comp)
        out_ready[x].record(comp)
        s_out.wait_event(out_ready[x])
        with torch.cuda.stream(s_out):
            h_out[x].copy_(d_out[x], non_blocking=True)
        out_free[x].record(s_out)

    def serial_step(k):
        d_in[0].copy_(h_ins[k % pools], non_blocking=True)
        api_call(k, 0)
        h_out[0].copy_(d_out[0], non_blocking=True)

    def timed(step, pipelined):
        for k in range(args.warmup):
            step(k)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        if pipelined:
            s_in.wait_event(e0)              # the first copy in starts inside the timed region
        for k in range(args.steps):
            step(k)
        if pipelined:
            comp.wait_stream(s_out)          # the last copy out ends inside it
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    pipe_ms = timed(pipelined_step, True)
    serial_ms = timed(serial_step, False)

    ref_bt = torch.from_numpy(base.block_tables).to(dev)
    ref_sl = torch.from_numpy(base.seq_lens).to(dev)
    ref_qsl = torch.from_numpy(base.query_start_loc).to(dev) if has_qsl else None
    ref_out, ref_lse = torch.empty_like(out), torch.empty_like(lse)
    nver = min(4, 2 * pools)
    same = True
    for k in range(nver):
        pipelined_step(k)
        comp.wait_stream(s_out)
        torch.cuda.synchronize()
        prepare(k % pools, works[k % pools].q, ref_bt, ref_sl, ref_qsl, ref_out, ref_lse)()
        torch.cuda.synchronize()
        x = k & 1
        same = same and torch.equal(h_oviews[x][0], ref_out.cpu()) and torch.equal(h_oviews[x][1], ref_lse.cpu())
    return pipe_ms, serial_ms, d_in[0].numel(), d_out[0].numel(), nver, same


def run_reference(args, world, rank):
    if rank != 0:
        return
    # every step one bounded sample, the whole run about --ref-total seconds of
    # oracle time (at most --ref-budget a step, at least one whole sequence)
    per_step = min(args.ref_budget, max(0.02, args.ref_total / (args.steps + args.warmup)))
    steps, cores, what = cpu_oracle_steps(args.config, [per_step] * (args.warmup + args.steps), threads=0, impl="c")
    timed = steps[args.warmup:]
    vals = [d["gbs"] for d in timed]
    sample = (f"{what}; {args.steps} timed samples after {args.warmup} warm-up ones, each about {per_step:.2f} s "
              f"of oracle time over whole sequences drawn from the {args.config} workload's length mix "
              f"(median {statistics.median([d['seqs'] for d in timed]):.0f} sequences, "
              f"{sum(d['tokens'] for d in timed)} cached tokens in all); value = median GB/s")
    from paged_kv_decode_06_gb300 import workloads as wl
    import numpy as np
    mla = args.config in wl.MLA_CONFIGS
    spec = wl.MLA_CONFIGS[args.config] if mla else wl.CONFIGS[args.config]
    sl, *_ = wl.draw_metadata(spec, np.random.default_rng(spec.seed))
    eb = 1 if spec.kv_dtype == "fp8" else 2
    if mla:
        step_bytes = int(sl.astype(np.int64).sum()) * spec.head_dim * eb
    else:
        per_row = spec.head_dim * eb + (4 if spec.token_scale_range is not None else 0)
        step_bytes = int(sl.astype(np.int64).sum()) * spec.num_kv_heads * 2 * per_row
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_bytes / (v * 1e9) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.config, "kv_bytes_per_step": step_bytes},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _setup_rank(local, world):
    import torch

    from paged_kv_decode_06_gb300 import binding
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl")
    binding.load()
    return dev


def measure_decode(spec, args, world, local, dev, window=0, sinks=False, tc=0):
    """Every timed pass of one grouped-query decode workload (see
    _timed_passes and _packed_e2e) plus the figures the JSON line reports."""
    import numpy as np
    import torch

    from paged_kv_decode_06_gb300 import binding
    from paged_kv_decode_06_gb300 import workloads as wl

    base = wl.make_workload(spec, device=str(dev))
    step_bytes = base.kv_bytes()
    sinks_t = None
    if window > 0:
        # algorithmic bytes with a sliding window: the union of the query rows'
        # windows, min(L, W + q - 1) keys per sequence
        eb = 1 if spec.kv_dtype == "fp8" else 2
        seen = np.minimum(base.seq_lens.astype(np.int64), window + base.query_lens.astype(np.int64) - 1)
        step_bytes = int(seen.sum()) * spec.num_kv_heads * spec.head_dim * 2 * eb
    if sinks:
        sinks_t = torch.randn(spec.num_q_heads, generator=torch.Generator().manual_seed(3)).to(dev)
    pools = min(16, max(1, math.ceil(2 * L2_BYTES / step_bytes)))
    # every pool shares the first one's metadata (lengths, page ids); only the contents differ
    works = [base] + [wl.make_workload(spec, device=str(dev), content_seed=spec.seed + 100 * k)
                      for k in range(1, pools)]

    def pool_options(w, **extra):
        # per-token fp8 scales belong to each pool's cache
        if window > 0 or sinks or tc or w.k_token_scales is not None or extra:
            return binding.make_options(sliding_window=window, sinks=sinks_t, use_tcgen05=tc,
                                        k_token_scales=w.k_token_scales, v_token_scales=w.v_token_scales, **extra)
        return None
    pool_opts = [pool_options(w) for w in works]
    bt = torch.from_numpy(base.block_tables).to(dev)
    sl = torch.from_numpy(base.seq_lens).to(dev)
    qsl = torch.from_numpy(base.query_start_loc).to(dev) if base.query_start_loc is not None else None
    mq = spec.max_query_len if qsl is not None else 1
    out = torch.empty_like(base.q)
    lse = torch.empty(base.q.shape[:2], dtype=torch.float32, device=dev)

    def step(k, opts=None, stream_=None):
        w = works[k % pools]
        if opts is None:
            opts = pool_opts[k % pools]
        binding.paged_attn_decode(w.q, w.k_cache, w.v_cache, bt, sl, qsl, mq, spec.scale, spec.k_scale,
                                  spec.v_scale, out=out, lse=lse, options=opts, stream=stream_)

    ms, split_ms, direct_ms, clocks, repeats = _timed_passes(
        step, lambda pidx, ea, eb: pool_options(works[pidx], split_start_event=ea, split_stop_event=eb), pools, args,
        world, local, dev)

    def e2e_prepare(pidx, q, bt_, sl_, qsl_, out_, lse_):
        w = works[pidx]
        return binding.prepare_decode(q, w.k_cache, w.v_cache, bt_, sl_, qsl_, mq, spec.scale, spec.k_scale,
                                      spec.v_scale, out=out_, lse=lse_, options=pool_opts[pidx])

    e2e_ms, e2e_serial_ms, h2d, d2h, e2e_nver, e2e_same = _packed_e2e(base, works, out, lse, dev, e2e_prepare, args)
    status = binding.paged_attn_device_status(clear=True)
    plan = binding.paged_attn_plan(spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                   binding.kv_dtype_code(spec.kv_dtype), mq,
                                   options=binding.make_options(use_tcgen05=tc))
    kernel = "pa_split_tc_kernel" if plan["variant"] == 1 else "pa_split_kernel"
    del works, base, out, lse
    torch.cuda.empty_cache()
    return dict(spec=spec, step_bytes=step_bytes, pools=pools, ms=ms, split_ms=split_ms, direct_ms=direct_ms,
                clocks=clocks, repeats=repeats, e2e_ms=e2e_ms, e2e_serial_ms=e2e_serial_ms, h2d=h2d, d2h=d2h,
                e2e_nver=e2e_nver, e2e_same=e2e_same,
                status=status, plan=plan,
                kernel=kernel, traffic=_traffic_from_profiles(spec.name, kernel), flops=None)


def measure_mla(spec, args, world, local, dev, tc=0):
    """measure_decode for MLA decode (paged_attn_mla_decode) on a latent cache
    [NB, 16, 576]: every cached row is read once per step."""
    import numpy as np
    import torch

    from paged_kv_decode_06_gb300 import binding
    from paged_kv_decode_06_gb300 import workloads as wl

    base = wl.make_mla_workload(spec, device=str(dev))
    step_bytes = base.kv_bytes()
    pools = min(16, max(1, math.ceil(2 * L2_BYTES / step_bytes)))
    works = [base] + [wl.make_mla_workload(spec, device=str(dev), content_seed=spec.seed + 100 * k)
                      for k in range(1, pools)]
    bt = torch.from_numpy(base.block_tables).to(dev)
    sl = torch.from_numpy(base.seq_lens).to(dev)
    qsl = torch.from_numpy(base.query_start_loc).to(dev) if base.query_start_loc is not None else None
    mq = spec.max_query_len if qsl is not None else 1
    T = base.q.shape[0]
    out = torch.empty((T, spec.num_q_heads, spec.kv_lora_rank), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, spec.num_q_heads), dtype=torch.float32, device=dev)

    kopts = binding.make_options(use_tcgen05=tc) if tc else None

    def step(k, opts=None, stream_=None):
        w = works[k % pools]
        binding.paged_attn_mla_decode(w.q, w.kv_cache, bt, sl, qsl, mq, spec.scale, spec.kv_scale, out=out, lse=lse,
                                      options=opts if opts is not None else kopts, stream=stream_)

    ev_opt = {}

    def ev_opts_for(pidx, ea, eb):
        if "o" not in ev_opt:
            ev_opt["o"] = binding.make_options(split_start_event=ea, split_stop_event=eb, use_tcgen05=tc)
        return ev_opt["o"]

    ms, split_ms, direct_ms, clocks, repeats = _timed_passes(step, ev_opts_for, pools, args, world, local, dev)

    def e2e_prepare(pidx, q, bt_, sl_, qsl_, out_, lse_):
        w = works[pidx]
        return binding.prepare_mla_decode(q, w.kv_cache, bt_, sl_, qsl_, mq, spec.scale, spec.kv_scale, out=out_,
                                          lse=lse_, options=kopts)

    e2e_ms, e2e_serial_ms, h2d, d2h, e2e_nver, e2e_same = _packed_e2e(base, works, out, lse, dev, e2e_prepare, args)
    status = binding.paged_attn_device_status(clear=True)
    plan = binding.paged_attn_mla_plan(spec.num_seqs, spec.num_q_heads, binding.kv_dtype_code(spec.kv_dtype), mq,
                                       options=binding.make_options(use_tcgen05=tc))
    # tensor work per step: 2 * rows * (576 + 512) flops per cached token of each row's sequence
    rows_tokens = int((base.seq_lens.astype(np.int64) * base.query_lens.astype(np.int64)).sum()) * spec.num_q_heads
    flops = 2 * rows_tokens * (spec.head_dim + spec.kv_lora_rank)
    del works, base, out, lse
    torch.cuda.empty_cache()
    kernel = "pa_mla_tc_kernel" if plan["variant"] == 3 else "pa_mla_kernel"
    return dict(spec=spec, step_bytes=step_bytes, pools=pools, ms=ms, split_ms=split_ms, direct_ms=direct_ms,
                clocks=clocks, repeats=repeats, e2e_ms=e2e_ms, e2e_serial_ms=e2e_serial_ms, h2d=h2d, d2h=d2h,
                e2e_nver=e2e_nver, e2e_same=e2e_same,
                status=status, plan=plan,
                kernel=kernel, traffic=_traffic_from_profiles(spec.name, kernel), flops=flops)


def _line(r, args, world, window=0, sinks=False, tc=0):
    """The JSON line of one measured workload (measure_decode / measure_mla)."""
    spec = r["spec"]
    peak, peak_kind = _peaks()
    split_mean = statistics.mean(r["split_ms"])
    achieved = r["step_bytes"] / (split_mean * 1e-3) / 1e9
    value = job_throughput_gbs(r["step_bytes"], world, r["ms"])
    mla = r["kernel"] in ("pa_mla_kernel", "pa_mla_tc_kernel")
    config = {"workload": spec.name, "num_seqs": spec.num_seqs, "q_heads": spec.num_q_heads}
    if mla:
        config.update(kv_lora_rank=spec.kv_lora_rank, rope_dim=spec.rope_dim, kv_dtype=spec.kv_dtype,
                      max_query_len=spec.max_query_len, flops_per_step=r["flops"])
    else:
        config.update(kv_heads=spec.num_kv_heads, head_dim=spec.head_dim, kv_dtype=spec.kv_dtype,
                      max_query_len=spec.max_query_len, sliding_window=window, sinks=bool(sinks), use_tcgen05=tc)
    api = "paged_attn_mla_decode" if mla else "paged_attn_decode"
    config.update({"kv_bytes_per_step": r["step_bytes"], "kv_pools_rotated": r["pools"],
                   "l2": "no flush; each step reads >= 2x L2 of KV (pools rotated when one is smaller)",
                   "step_mode": f"CUDA graph replay; a step = one {api} call (split + merge)",
                   "timed_windows": f"{r['repeats']} windows of exactly {args.steps} steps; value from the median "
                                    f"window",
                   "plan": r["plan"]})
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": r["traffic"], "kernel": r["kernel"], "peak_source": f"{peak_kind} hbm_gbs",
            "split_kernel_us_mean": split_mean * 1e3, "split_kernel_us_median": statistics.median(r["split_ms"]) * 1e3,
            "per_launch_bytes": r["step_bytes"]}
    if mla:
        roof["tensor_tflops"] = r["flops"] / (split_mean * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"], "us_per_step": r["ms"] * 1e3,
        "frac_of_hbm_peak": value / world / peak, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f8e4m3" if spec.kv_dtype == "fp8" else "bf16", "data": "synthetic",
        "config": config, "roofline": roof,
        "e2e": {"value": r["step_bytes"] / (min(r["e2e_ms"], r["e2e_serial_ms"]) * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": min(r["e2e_ms"], r["e2e_serial_ms"]),
                "schedule": "pipelined" if r["e2e_ms"] <= r["e2e_serial_ms"] else "serial",
                "pipelined_value": r["step_bytes"] / (r["e2e_ms"] * 1e-3) / 1e9, "pipelined_ms_per_step": r["e2e_ms"],
                "serial_value": r["step_bytes"] / (r["e2e_serial_ms"] * 1e-3) / 1e9,
                "serial_ms_per_step": r["e2e_serial_ms"],
                "verified_steps": r["e2e_nver"], "verified_equal_to_direct_call": r["e2e_same"],
                "note": "per step: one copy of the packed inputs from pinned host memory, the API call from "
                        "Python (a prepared call: arguments marshalled once, the buffers refreshed in place), "
                        "one copy of the packed out / lse back, in two schedules: pipelined (the copies "
                        "of steps k + 1 and k - 1 on their own streams while step k computes, device buffers "
                        "double-buffered) and serial (copy in, call, copy out in order on one stream); value is "
                        "the faster (short steps are bound by the host's per-call work, which the pipelined "
                        "schedule's stream and event calls add to)"},
        "direct_call": {"value": r["step_bytes"] * world / (r["direct_ms"] * 1e-3) / 1e9, "unit": "GB/s",
                        "ms_per_step": r["direct_ms"],
                        "note": f"{api} called from Python each step (no CUDA graph)"},
        "gpu_launches": 2 * args.steps * r["repeats"],   # split + merge per timed step
        "clocks": r["clocks"],
        "device_status": r["status"],
    }


# Workloads measured beside the headline one in the same process (their
# `per_config` entries): the other decode configurations, then the extensions.
PER_CONFIG = ["tiny", "batch1_32k", "fp8", "mtp", "verify8", "fp8_pertoken", "mla_tp8", "mla_mtp_fp8"]


def _per_config_entry(r, args, world):
    ln = _line(r, args, world)
    roof = ln["roofline"]
    return {"us_per_step": ln["us_per_step"], "kv_gbs": ln["value"], "frac": ln["frac_of_hbm_peak"],
            "split_kernel_us": roof["split_kernel_us_mean"], "split_kernel_frac": roof["frac"],
            "traffic": roof["traffic"], "kernel": roof["kernel"], "kv_bytes_per_step": r["step_bytes"],
            "e2e_gbs": ln["e2e"]["value"], "e2e_schedule": ln["e2e"]["schedule"],
            "e2e_pipelined_gbs": ln["e2e"]["pipelined_value"], "e2e_serial_gbs": ln["e2e"]["serial_value"],
            "e2e_verified": ln["e2e"]["verified_equal_to_direct_call"],
            "timed_windows": r["repeats"], "clocks": ln["clocks"],
            "device_status": r["status"], "dtype": ln["dtype"]}


def run_ours(args, world, rank, local):
    import torch

    from paged_kv_decode_06_gb300 import workloads as wl
    dev = _setup_rank(local, world)
    mla = args.config in wl.MLA_CONFIGS
    if mla:
        spec = wl.MLA_CONFIGS[args.config]
        if args.batch:
            import dataclasses
            spec = dataclasses.replace(spec, num_seqs=args.batch, name=f"{spec.name}_b{args.batch}")
        r = measure_mla(spec, args, world, local, dev, tc=args.tc)
    else:
        spec = _spec_for(args)
        r = measure_decode(spec, args, world, local, dev, window=args.window, sinks=args.sinks, tc=args.tc)
    per_config = {}
    if not args.no_per_config and not args.batch and args.window == 0 and not args.sinks and args.tc == 0:
        for name in PER_CONFIG:
            if name == args.config:
                continue
            if name in wl.MLA_CONFIGS:
                pr = measure_mla(wl.MLA_CONFIGS[name], args, world, local, dev)
            else:
                pr = measure_decode(wl.CONFIGS[name], args, world, local, dev)
            per_config[name] = _per_config_entry(pr, args, world)
    if rank == 0:
        line = _line(r, args, world, window=args.window, sinks=args.sinks, tc=args.tc)
        if per_config:
            line["per_config"] = per_config
            line["gpu_launches"] += sum(2 * args.steps * e["timed_windows"] for e in per_config.values())
        if not args.no_cpu_baseline and not args.batch:
            line["cpu_baseline"] = cpu_baseline(args.config, args.cpu_budget)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_cache_write(args, world, rank, local):
    """Throughput of paged_attn_cache_write: one step writes the K and V rows of
    T new tokens (a prefill chunk of max_num_batched_tokens = 16384 tokens by
    default) into randomly permuted page slots.  Bytes = rows read (bf16) +
    rows written (cache dtype)."""
    import numpy as np
    import torch

    from paged_kv_decode_06_gb300 import binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()
    T, Hkv, D = args.tokens, 8, 128
    fp8 = args.kv_dtype == "fp8"
    esz = 1 if fp8 else 2
    NB = (T + 15) // 16 + 64
    g = torch.Generator(device=dev).manual_seed(77)
    key = torch.randn(T, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
    val = torch.randn(T, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
    cdt = torch.uint8 if fp8 else torch.bfloat16
    kc = torch.zeros(NB, 16, Hkv, D, dtype=cdt, device=dev)
    vc = torch.zeros(NB, 16, Hkv, D, dtype=cdt, device=dev)
    slots = torch.from_numpy(np.random.default_rng(5).permutation(NB * 16)[:T].astype(np.int32)).to(dev)
    ks = vs = 0.05 if fp8 else 1.0
    per_token = bool(args.per_token)
    if per_token and not fp8:
        raise SystemExit("--per-token needs --kv-dtype fp8")
    step_bytes = T * Hkv * D * 2 * (2 + esz) + (T * Hkv * 2 * 4 if per_token else 0)   # + the row scales
    # pools rotated so a step's bytes exceed 2x L2
    pools = max(1, math.ceil(2 * L2_BYTES / step_bytes))
    keys = [key] + [torch.randn_like(key, dtype=torch.float32).to(torch.bfloat16) for _ in range(pools - 1)]
    vals = [val] + [torch.randn_like(val, dtype=torch.float32).to(torch.bfloat16) for _ in range(pools - 1)]
    caches = [(kc, vc)] + [(torch.zeros_like(kc), torch.zeros_like(vc)) for _ in range(pools - 1)]
    scales = [(torch.zeros(NB, Hkv, 16, device=dev), torch.zeros(NB, Hkv, 16, device=dev)) for _ in range(pools)]
    stream = torch.cuda.current_stream()

    def write(key_, val_, c, sc, stream_=None):
        if per_token:
            binding.paged_attn_cache_write_per_token(key_, val_, slots, c[0], c[1], sc[0], sc[1], stream=stream_)
        else:
            binding.paged_attn_cache_write(key_, val_, slots, c[0], c[1], ks, vs, stream=stream_)

    def step(k, stream_=None):
        write(keys[k % pools], vals[k % pools], caches[k % pools], scales[k % pools], stream_)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    gsteps = pools * max(1, 8 // pools)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for j in range(gsteps):
            step(j, stream_=cap)
    singles = []
    for pidx in range(pools):
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg, stream=cap):
            step(pidx, stream_=cap)
        singles.append(gg)
    graph.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        t0.record(stream)
        k = 0
        while k + gsteps <= args.steps:
            graph.replay()
            k += gsteps
        while k < args.steps:
            singles[k % pools].replay()
            k += 1
        t1.record(stream)
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    # e2e: new rows copied in from pinned host memory each step
    hk = key.cpu().pin_memory()
    hv = val.cpu().pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(max(1, args.steps // 10)):
        key.copy_(hk, non_blocking=True)
        val.copy_(hv, non_blocking=True)
        write(key, val, (kc, vc), scales[0])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / max(1, args.steps // 10)
    peak, peak_kind = _peaks()
    value = step_bytes / (ms * 1e-3) / 1e9
    workload = f"cache_write_T{T}_{args.kv_dtype}" + ("_per_token" if per_token else "")
    kernel = "pa_cache_write_tok_kernel" if per_token else "pa_cache_write_kernel"
    line = {
        "metric": "paged KV cache write GB/s (rows read + written), 1 GPU", "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f8e4m3" if fp8 else "bf16", "data": "synthetic",
        "config": {"workload": workload,
                   "tokens": T, "kv_heads": Hkv, "head_dim": D,
                   "bytes_per_step": step_bytes, "pools_rotated": pools,
                   "step_mode": "CUDA graph replay of paged_attn_cache_write"},
        "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "traffic": _traffic_from_profiles(workload, kernel), "kernel": kernel,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": 2 * key.numel() * 2, "d2h_bytes_per_step": 0},
        "gpu_launches": args.steps, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def _spec_for(args):
    import dataclasses

    from paged_kv_decode_06_gb300 import workloads as wl
    spec = wl.CONFIGS[args.config]
    if args.batch:
        spec = dataclasses.replace(spec, num_seqs=args.batch, name=f"{spec.name}_b{args.batch}")
    return spec


def kernel_source_sha256(kernel):
    """Hash of the sources a kernel is compiled from (stamps ncu figures)."""
    import hashlib
    if kernel.startswith("pa_cache_write"):
        names = ["pa_cache_write.cu", "pa_device.cuh", "pa_pack.cuh"]
    else:
        names = ["pa_split.cuh", "pa_device.cuh", "pa_pack.cuh"] + \
            (["pa_split_tc.cuh"] if kernel == "pa_split_tc_kernel" else []) + \
            (["pa_mla.cu"] if kernel == "pa_mla_kernel" else []) + \
            (["pa_split_tc.cuh", "pa_mla_tc.cu"] if kernel == "pa_mla_tc_kernel" else [])
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_decode_06_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic_from_profiles(config, kernel):
    """DRAM bytes per launch of a kernel from the committed ncu summary, when it
    was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    entry = d.get(config)
    if not entry or entry.get("kernel") != kernel or entry.get("kernel_source_sha256") != kernel_source_sha256(kernel):
        return None
    return entry.get("dram_bytes_per_launch")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="llama3_8b")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch size (profiling cases)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="decode", choices=["decode", "cache_write"])
    ap.add_argument("--window", type=int, default=0, help="decode: sliding window of W keys (0 = off)")
    ap.add_argument("--sinks", action="store_true", help="decode: per-query-head attention sinks")
    ap.add_argument("--tc", type=int, default=0, choices=[0, 1, 2],
                    help="split kernel: 0 planner's choice, 1 mma.sync, 2 tcgen05 (grouped-query: bf16 caches)")
    ap.add_argument("--tokens", type=int, default=16384, help="cache_write: tokens written per step")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"], help="cache_write: cache dtype")
    ap.add_argument("--per-token", action="store_true", help="cache_write: fp8 with one scale per row")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="decode: repeat the K-step timed window until the windows add up to this long")
    ap.add_argument("--no-per-config", action="store_true",
                    help="decode: measure only --config (no per_config entries for the other workloads)")
    ap.add_argument("--ref-budget", type=float, default=8.0, help="reference arm: most oracle seconds a step")
    ap.add_argument("--ref-total", type=float, default=120.0,
                    help="reference arm: oracle seconds of the whole run (split over warm-up and timed steps)")
    args = ap.parse_args()
    world, rank, local = _dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.op == "cache_write":
        run_cache_write(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
