"""Benchmark of the causal kernelized linear attention library on GB300.

One JSON line on rank 0.  Headline: the causal forward of the long-sequence
workload (B=1, H=16, n=65536, d=d'=128, bf16 inputs, elu+1, per-head decay
a ~ U[0.95, 0.9999], fp32 state) — the n ≥ 16K configuration at which the
forward metric is quoted.  A step is one la_forward over the whole batch.
Secondary lines (same JSON object, key "secondary") time the other
workloads: elu+1 with decay at n=2048, Performer (m=256) causal and
non-causal, non-causal elu+1 (eq (6)) at the n=2048 and the long shape, the
long shape with a per-token decay and input weight, the backward, and the
recurrent decode step (B=256, H=32, d=128; and Performer, d=64, m=256).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs an independent
replica of the workload (the heads are independent; no collective is on the
data path), "scaling": "weak"; value = tokens of all ranks / max rank time.
``--impl reference`` times the fp64 CPU oracle (the only reference that
exists for this method) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "causal linear-attn fwd tokens/s & TFLOP/s (% bf16 peak); decode-step GB/s (% HBM)"
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- helpers

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel source still matches the one the counters were taken on."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get(kernel_key)
    if not t:
        return None
    try:
        if _source_sha(t["sources"]) != t["sources_sha"]:
            return None
    except OSError:
        return None
    return t["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.lines = []
        self.proc = None
        self.dev = device_index

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _time_steps(fn, steps, warmup, stream, flush=None, counter=None):
    """Per-step device time (ms) with CUDA events on the launching stream, and
    the number of library launches queued inside the timed steps."""
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    launches = 0
    for i in range(steps):
        if flush is not None:
            flush()
        c0 = counter() if counter else 0
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
        launches += (counter() - c0) if counter else 0
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], launches


def _max_over_ranks(x, dist):
    """The largest x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(units_per_rank, seconds, world, dist):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time."""
    return units_per_rank * world / _max_over_ranks(seconds, dist)


def _barrier(dist):
    if dist is not None:
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


# ----------------------------------------------------------------------------- workloads

def _fwd_alg(w: W.ForwardWorkload):
    """Algorithmic work of one forward over the batch: flops 4·d'·d + 4·d' per
    token-head (+ 4·d·m for the two Performer projections), bytes = q, k, v
    read + o written."""
    th = w.B * w.H * w.n
    dp = w.dprime
    flops = th * (4 * dp * w.d + 4 * dp + (4 * w.d * w.m if w.feature_map == "performer" else 0))
    esize = 2 if w.dtype == "bf16" else 4
    nbytes = th * w.d * esize * 4
    return flops, nbytes


def bench_forward(cl, w, causal, steps, warmup, stream, flush_l2, peaks, want_e2e=False):
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.forward_inputs(w)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty_like(g["q"])
    fm = w.feature_map

    def step():
        cl.forward(g["q"], g["k"], g["v"], g["a"], fm, g["omega"], causal, out=out, stream=stream)

    flush = None
    if flush_l2:
        buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        flush = lambda: buf.fill_(1.0)  # noqa: E731
    ms, launches = _time_steps(step, steps, warmup, stream, flush, cl.launch_count)
    flops, nbytes = _fwd_alg(w)
    avg_ms = statistics.mean(ms)
    res = {"ms": ms, "avg_ms": avg_ms, "flops": flops, "bytes": nbytes,
           "launches_per_step": launches / steps, "launches_timed": launches,
           "tokens": w.B * w.n}
    if want_e2e:
        res["e2e"] = bench_forward_e2e(cl, w, causal, inp, steps, warmup, stream)
    return res


def bench_shard_rank(cl, w: W.ForwardWorkload, nshards, steps, warmup, stream):
    """One rank's work in the sequence-sharded causal forward of workload w
    split into nshards equal shards, on this GPU: the aggregate of its shard
    (la_forward_state), the state entering it from the gathered aggregates of
    all shards (la_shard_entering_state) and its outputs from that state
    (la_forward_from_state).  The all-gathers between the steps are not
    timed (one GPU).  The last rank is timed (its entering state combines
    every earlier shard)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    L = w.n // nshards
    inp = W.forward_inputs(w)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    r = nshards - 1
    q, k, v = (g[x][:, :, r * L:(r + 1) * L].contiguous() for x in ("q", "k", "v"))
    dp = w.dprime
    gathered = torch.zeros(nshards, w.B * w.H * (dp * w.d + dp), device=dev, dtype=torch.float32)
    mu_a = gathered[r, :w.B * w.H * dp * w.d].view(w.B, w.H, dp, w.d)
    nu_a = gathered[r, w.B * w.H * dp * w.d:].view(w.B, w.H, dp)
    out = torch.empty_like(q)

    def step():
        cl.forward_state(k, v, g["a"], w.feature_map, g["omega"], mu_out=mu_a, nu_out=nu_a,
                         stream=stream)
        mu_in, nu_in = cl.shard_entering_state(gathered, r, [L] * nshards, w.B, w.H, dp, w.d,
                                               g["a"], stream=stream)
        cl.forward_from_state(q, k, v, mu_in, nu_in, g["a"], w.feature_map, g["omega"], out=out,
                              stream=stream)

    ms, launches = _time_steps(step, steps, warmup, stream, None, cl.launch_count)
    avg_ms = statistics.mean(ms)
    nbytes = w.B * w.H * L * w.d * 2 * 4
    return {"ms": ms, "avg_ms": avg_ms, "tokens": w.B * L, "bytes": nbytes,
            "launches_per_step": launches / steps}


def bench_token_decay(cl, tw: W.TokenDecayWorkload, steps, warmup, stream):
    """la_forward_token_decay over the whole batch: per-token a and b [B,H,n]
    fp32.  Algorithmic bytes: q, k, v read and o written (bf16) plus a and b
    read (fp32) per token-head."""
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.token_decay_inputs(tw)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty_like(g["q"])
    w = tw.base

    def step():
        cl.forward_token_decay(g["q"], g["k"], g["v"], g["a_tok"], g["b_tok"], "elu1", None,
                               out=out, stream=stream)

    ms, launches = _time_steps(step, steps, warmup, stream, None, cl.launch_count)
    th = w.B * w.H * w.n
    flops, nbytes = _fwd_alg(w)
    nbytes += th * 4 * (2 if tw.weight else 1)
    return {"ms": ms, "avg_ms": statistics.mean(ms), "flops": flops, "bytes": nbytes,
            "launches_per_step": launches / steps, "tokens": w.B * w.n}


def bench_backward(cl, w: W.ForwardWorkload, steps, warmup, stream):
    """la_backward over the whole batch (∂q, ∂k, ∂v and ∂a of the causal
    forward).  Algorithmic bytes: q, k, v, ∂o read and ∂q, ∂k, ∂v written."""
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.forward_inputs(w)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    gen = torch.Generator().manual_seed(w.seed + 1000)
    go = torch.randn(w.B, w.H, w.n, w.d, generator=gen).to(W.torch_dtype(w.dtype)).to(dev)
    dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))

    def step():
        cl.backward(g["q"], g["k"], g["v"], go, g["a"], w.feature_map, g["omega"], dq=dq, dk=dk,
                    dv=dv, stream=stream)

    ms, launches = _time_steps(step, steps, warmup, stream, None, cl.launch_count)
    esize = 2 if w.dtype == "bf16" else 4
    nbytes = w.B * w.H * w.n * w.d * esize * 7
    return {"ms": ms, "avg_ms": statistics.mean(ms), "bytes": nbytes,
            "launches_per_step": launches / steps, "tokens": w.B * w.n}


def bench_forward_e2e(cl, w, causal, inp, steps, warmup, stream):
    """Same forward through the public API with host buffers: every step copies
    its q, k, v from pinned host memory, runs la_forward and copies o back to
    pinned host memory.  The copies run on their own streams (one per tensor)
    with two device buffer sets, so that step i's input copies and step i−1's output copy
    overlap step i−1's and step i's compute (stream order and events keep every
    buffer's uses in sequence).  One event pair spans all the timed steps; the
    per-step time is that span / steps."""
    dev = torch.device("cuda", torch.cuda.current_device())
    hq, hk, hv = (inp[k].pin_memory() for k in ("q", "k", "v"))
    hout = torch.empty_like(inp["q"]).pin_memory()
    dbuf = [[torch.empty_like(x, device=dev) for x in (hq, hk, hv)] + [torch.empty_like(hq, device=dev)]
            for _ in range(2)]
    a = inp["a"].to(dev) if inp["a"] is not None else None
    om = inp["omega"].to(dev) if inp["omega"] is not None else None
    s_in = [torch.cuda.Stream(device=dev) for _ in range(3)]   # one per input: q, k, v
    s_out = torch.cuda.Stream(device=dev)
    in_done = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        dq, dk, dv, dout = dbuf[b]
        for j, (dst, src) in enumerate(((dq, hq), (dk, hk), (dv, hv))):
            s_in[j].wait_event(comp_done[b])     # step i−2's compute has read this set
            with torch.cuda.stream(s_in[j]):
                dst.copy_(src, non_blocking=True)
            in_done[b][j].record(s_in[j])
            stream.wait_event(in_done[b][j])
        stream.wait_event(out_done[b])           # step i−2's output has been copied out
        cl.forward(dq, dk, dv, a, w.feature_map, om, causal, out=dout, stream=stream)
        comp_done[b].record(stream)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            hout.copy_(dout, non_blocking=True)
        out_done[b].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for si in s_in:
        si.wait_event(t0)
    s_out.wait_event(t0)
    for i in range(steps):
        step(i)
    stream.wait_event(out_done[(steps - 1) % 2])
    t1.record(stream)
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size()
    return {"ms": [total / steps] * steps, "h2d": h2d, "d2h": d2h,
            "overlap": "q, k, v and o copies on four streams overlap compute; two device buffer sets"}


def bench_forward_host(cl, w, causal, inp, steps, warmup, stream):
    """The same forward through la_forward_host: q, k, v in pinned host memory
    go in and o comes back inside one library call per step (the library
    cuts the sequence into pieces whose copies overlap the compute of the
    others).  One event pair spans the timed calls."""
    pin = {k: (x.pin_memory() if isinstance(x, torch.Tensor) else x) for k, x in inp.items()}
    out = torch.empty_like(inp["q"]).pin_memory()

    def step():
        cl.forward_host(pin["q"], pin["k"], pin["v"], pin["a"], w.feature_map, pin["omega"],
                        causal, out=out, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def bench_decode(cl, w: W.DecodeWorkload, stream, steps=None, distinct=32):
    """Prefill through la_forward_with_state, then `steps` decode steps (one
    launch each); per-step q, k, v cycle over `distinct` pre-generated sets."""
    dev = torch.device("cuda", torch.cuda.current_device())
    steps = steps or w.steps
    pre = W.decode_prefill_inputs(w)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in pre.items()}
    _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], w.feature_map, g["omega"],
                                      stream=stream)
    del g["q"], g["k"], g["v"]
    sets = []
    for s in range(distinct):
        st = W.decode_step_inputs(w, s)
        sets.append({k: v.to(dev) for k, v in st.items()})
    out = torch.empty(w.B, w.H, w.d, device=dev, dtype=torch.bfloat16)
    it = [0]

    def step():
        x = sets[it[0] % distinct]
        it[0] += 1
        cl.decode_step(mu, nu, x["q"], x["k"], x["v"], g["a"], out=out, stream=stream,
                       feature_map=w.feature_map, omega=g["omega"])

    ms, launches = _time_steps(step, steps, 3, stream, None, cl.launch_count)
    heads = w.B * w.H
    # algorithmic bytes per head-step: μ read+write 8·d'·d, ν read+write 8·d',
    # q, k, v read and o written in bf16 (8·d); ω (Performer) is shared by all
    # heads and read once per step
    dp = w.m if w.feature_map == "performer" else w.d
    nbytes = heads * (8 * dp * w.d + 8 * dp + 8 * w.d) + 2 * w.d * w.m
    return {"ms": ms, "avg_ms": statistics.mean(ms), "bytes": nbytes, "tokens": w.B,
            "launches_timed": launches}


# ----------------------------------------------------------------------------- CPU oracle

def cpu_oracle_sample(w: W.ForwardWorkload, causal=True, target_s=12.0):
    """Time the fp64 oracle on a bounded prefix of the workload (all heads,
    the first n_s tokens); the per-token cost of the recurrence does not
    depend on the position, so tokens/s of the prefix is that of the whole."""
    import oracle
    oracle.build()
    n_s = 64
    while True:
        inp = W.forward_inputs(w, n=n_s)
        t0 = time.perf_counter()
        oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], w.feature_map, inp["omega"], causal)
        dt = time.perf_counter() - t0
        if dt >= target_s or n_s >= w.n:
            break
        n_s = min(w.n, max(n_s * 2, int(n_s * target_s / max(dt, 1e-3) * 0.9)))
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    cores = min(threads, w.B * w.H)
    # one core: a single head (the oracle parallelises over heads only)
    n_1 = 64
    while True:
        inp = W.forward_inputs(w, n=n_1)
        one = {k: (x[:1, :1].contiguous() if k in ("q", "k", "v") else x) for k, x in inp.items()}
        a1 = one["a"][:1] if one["a"] is not None else None
        t0 = time.perf_counter()
        oracle.forward(one["q"], one["k"], one["v"], a1, w.feature_map, one["omega"], causal)
        dt1 = time.perf_counter() - t0
        if dt1 >= target_s / 4 or n_1 >= w.n:
            break
        n_1 = min(w.n, max(n_1 * 2, int(n_1 * target_s / 4 / max(dt1, 1e-3) * 0.9)))
    return {"value": w.B * n_s / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"all {w.B * w.H} heads x first {n_s} of {w.n} tokens "
                      f"(fp64 per-token recurrence, OpenMP over heads), {dt:.1f} s",
            "single_core": {"value": n_1 / dt1 / w.H, "unit": "tokens/s", "cores": 1,
                            "sample": f"head 0 of batch 0, first {n_1} tokens, {dt1:.1f} s; "
                                      f"head-tokens/s divided by the {w.H} heads of a token"}}


# ----------------------------------------------------------------------------- arms

def run_reference(args, rank):
    """--impl reference: the fp64 CPU oracle on bounded samples of the headline
    workload, one sample per step."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = W.LONG
    n_s = 128
    for _ in range(args.warmup):
        inp = W.forward_inputs(w, n=n_s)
        oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], "elu1", None, True)
    inp = W.forward_inputs(w, n=n_s)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(inp["q"], inp["k"], inp["v"], inp["a"], "elu1", None, True)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = w.B * n_s * args.steps / tot
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    cores = min(threads, w.B * w.H)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "d": w.d,
                       "feature_map": "elu1", "causal": True, "decay": list(w.decay),
                       "sample_tokens_per_head": n_s},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"all {w.B * w.H} heads x first {n_s} tokens per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, rank, world, dist):
    import causal_kernelized_linear_gb300 as cl
    cl.build()
    cl.load()
    dev = torch.cuda.current_device()
    stream = torch.cuda.current_stream()
    peaks = _peaks()
    w = W.LONG

    sampler = ClockSampler(dev) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    _barrier(dist)
    main = bench_forward(cl, w, True, args.steps, args.warmup, stream, flush_l2=False, peaks=peaks,
                         want_e2e=not args.no_e2e)
    _barrier(dist)
    clocks = sampler.stop() if sampler else None

    step_s = _max_over_ranks(sum(main["ms"]) / 1e3, dist)
    value = _job_rate(w.B * w.n * args.steps, step_s, world, None)
    ms_per_step = 1e3 * step_s / args.steps
    tflops = main["flops"] / (ms_per_step / 1e3) / 1e12
    achieved = main["bytes"] / (main["avg_ms"] / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": "la_forward (whole call)", "achieved": achieved,
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "traffic": _traffic("forward_long"), "peak_source": peaks["source"],
            "algorithmic_bytes_per_launch": main["bytes"]}
    e2e = None
    if "e2e" in main:
        e_s = _max_over_ranks(sum(main["e2e"]["ms"]) / 1e3, dist)
        e2e = {"value": _job_rate(w.B * w.n * args.steps, e_s, world, None), "unit": "tokens/s",
               "h2d_bytes_per_step": main["e2e"]["h2d"], "d2h_bytes_per_step": main["e2e"]["d2h"],
               "pipelining": main["e2e"]["overlap"],
               "ms_per_step": 1e3 * e_s / args.steps}
        # the same through the library's host-buffer entry point
        h_ms = bench_forward_host(cl, w, True, W.forward_inputs(w), args.steps, args.warmup,
                                  stream)
        e2e["host_api"] = {"call": "la_forward_host", "value": w.B * w.n / (h_ms / 1e3),
                           "unit": "tokens/s", "ms_per_step": h_ms,
                           "h2d_bytes_per_step": main["e2e"]["h2d"],
                           "d2h_bytes_per_step": main["e2e"]["d2h"]}

    secondary = []
    if not args.no_secondary:
        for sw, causal, flush in ((W.ELU1_DECAY, True, True), (W.PERFORMER, False, True),
                                  (W.PERFORMER, True, True), (W.ELU1_NONCAUSAL, False, True),
                                  (W.LONG_NONCAUSAL, False, False)):
            r = bench_forward(cl, sw, causal, max(args.steps, 20), max(args.warmup, 3), stream,
                              flush_l2=flush, peaks=peaks)
            secs = r["avg_ms"] / 1e3
            fl = r["flops"] / secs / 1e12
            gbs = r["bytes"] / secs / 1e9
            secondary.append({
                "workload": sw.name, "causal": causal, "value": sw.B * sw.n / secs,
                "unit": "tokens/s", "ms_per_step": r["avg_ms"], "tflops_alg": fl,
                "frac_bf16_peak": fl / peaks["bf16_tflops"], "gbs_alg": gbs,
                "frac_hbm": gbs / peaks["hbm_gbs"],
                "l2": "flushed between steps" if flush else "inputs (805 MiB) larger than L2",
                "launches_per_step": r["launches_per_step"]})
        tw = W.TOKEN_DECAY_LONG
        r = bench_token_decay(cl, tw, max(args.steps, 20), max(args.warmup, 3), stream)
        secs = r["avg_ms"] / 1e3
        gbs = r["bytes"] / secs / 1e9
        fl = r["flops"] / secs / 1e12
        secondary.append({
            "workload": tw.name, "causal": True, "value": r["tokens"] / secs, "unit": "tokens/s",
            "ms_per_step": r["avg_ms"], "tflops_alg": fl,
            "frac_bf16_peak": fl / peaks["bf16_tflops"], "gbs_alg": gbs,
            "frac_hbm": gbs / peaks["hbm_gbs"],
            "decay": "per token: a = exp(-A_h*softplus(z-4)), b = softplus(z-4)",
            "l2": "inputs (776 MiB) larger than L2; no flush",
            "launches_per_step": r["launches_per_step"]})
        for bw in (W.ELU1_DECAY, W.LONG):
            r = bench_backward(cl, bw, 5 if bw is W.LONG else max(args.steps, 20), 3, stream)
            secs = r["avg_ms"] / 1e3
            gbs = r["bytes"] / secs / 1e9
            secondary.append({
                "workload": bw.name, "pass": "backward (dq, dk, dv, da; tcgen05 tensor cores, bf16 operands, fp32 state)",
                "value": r["tokens"] / secs, "unit": "tokens/s", "ms_per_step": r["avg_ms"],
                "gbs_alg": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "steps": len(r["ms"]),
                "launches_per_step": r["launches_per_step"]})
        r = bench_shard_rank(cl, W.LONG, 2, max(args.steps, 20), max(args.warmup, 3), stream)
        secs = r["avg_ms"] / 1e3
        gbs = r["bytes"] / secs / 1e9
        secondary.append({
            "workload": W.LONG.name, "pass": "sequence-sharded forward, one rank of 2 (n/2 tokens): "
            "state pass, entering state, forward from it; all-gathers not included (one GPU)",
            "value": r["tokens"] / secs, "unit": "tokens/s (this rank)", "ms_per_step": r["avg_ms"],
            "gbs_alg": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
            "l2": "inputs (403 MiB) larger than L2; no flush",
            "launches_per_step": r["launches_per_step"]})
        for dw in (W.DECODE, W.PERFORMER_DECODE):
            d = bench_decode(cl, dw, stream)
            secs = d["avg_ms"] / 1e3
            gbs = d["bytes"] / secs / 1e9
            secondary.append({
                "workload": dw.name, "value": gbs, "unit": "GB/s",
                "frac_hbm": gbs / peaks["hbm_gbs"], "tokens_per_s": d["tokens"] * dw.H / secs,
                "ms_per_step": d["avg_ms"], "steps": len(d["ms"]),
                "l2": "state (512 MiB) larger than L2",
                "launches_per_step": 1})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(w, True, target_s=args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "d": w.d,
                           "dprime": w.dprime, "feature_map": "elu1", "causal": True,
                           "decay": list(w.decay), "state_dtype": "f32",
                           "l2": "inputs (768 MiB) larger than L2; no flush",
                           "parallelism": f"replicas x{world}"},
                "tflops_alg": tflops, "frac_bf16_peak": tflops / peaks["bf16_tflops"],
                "roofline": roof, "e2e": e2e, "gpu_launches": main["launches_timed"],
                "clocks": clocks, "cpu_baseline": cpu, "secondary": secondary}
        print(json.dumps(line), flush=True)
    return 0


def run_profile_case(case):
    """Small seeded cases for ncu captures: a few calls of one entry point,
    sized so that a full capture ends in about a minute (inputs larger than
    L2, a few hundred MB on the device)."""
    import causal_kernelized_linear_gb300 as cl
    cl.build()
    cl.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if case == "forward-long-small":
        w = W.LONG
        inp = W.forward_inputs(w, n=32768)          # B1 H16 n32768 d128: 512 MiB of q, k, v, o
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        out = torch.empty_like(g["q"])
        for _ in range(3):
            cl.forward(g["q"], g["k"], g["v"], g["a"], "elu1", None, True, out=out)
    elif case == "noncausal-long-small":
        w = W.LONG_NONCAUSAL
        inp = W.forward_inputs(w, n=32768)          # B1 H16 n32768 d128: 512 MiB of q, k, v, o
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        out = torch.empty_like(g["q"])
        for _ in range(3):
            cl.forward(g["q"], g["k"], g["v"], None, "elu1", None, False, out=out)
    elif case == "elu1-decay":
        w = W.ELU1_DECAY                             # B4 H8 n2048 d64 (the workload itself)
        inp = W.forward_inputs(w)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        out = torch.empty_like(g["q"])
        for _ in range(3):
            cl.forward(g["q"], g["k"], g["v"], g["a"], "elu1", None, True, out=out)
    elif case == "performer":
        w = W.PERFORMER                              # B2 H8 n4096 d64 m256 (the workload itself)
        inp = W.forward_inputs(w)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        out = torch.empty_like(g["q"])
        for causal in (True, False):
            for _ in range(3):
                cl.forward(g["q"], g["k"], g["v"], None, "performer", g["omega"], causal, out=out)
    elif case == "performer-decode-small":
        w = W.PERFORMER_DECODE
        B = 64                                       # B64 H32 d64 m256: 128 MiB of state
        pre = W.decode_prefill_inputs(w, B=B)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in pre.items()}
        _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "performer", g["omega"])
        for step in range(5):
            st = {k: v.to(dev) for k, v in W.decode_step_inputs(w, step, B=B).items()}
            cl.decode_step(mu, nu, st["q"], st["k"], st["v"], g["a"], feature_map="performer",
                           omega=g["omega"])
    elif case == "token-decay-small":
        tw = W.TOKEN_DECAY_LONG
        inp = W.token_decay_inputs(tw, n=32768)     # B1 H16 n32768 d128 + a, b: 516 MiB
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        out = torch.empty_like(g["q"])
        for _ in range(3):
            cl.forward_token_decay(g["q"], g["k"], g["v"], g["a_tok"], g["b_tok"], "elu1", None,
                                   out=out)
    elif case == "backward-small":
        w = W.ELU1_DECAY                             # B4 H8 n2048 d64 (the workload itself)
        inp = W.forward_inputs(w)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        gen = torch.Generator().manual_seed(w.seed + 1000)
        go = torch.randn(w.B, w.H, w.n, w.d, generator=gen).bfloat16().to(dev)
        for _ in range(3):
            cl.backward(g["q"], g["k"], g["v"], go, g["a"], "elu1")
    elif case == "backward-long-small":
        w = W.LONG
        inp = W.forward_inputs(w, n=16384)          # B1 H16 n16384 d128: 64 MiB per tensor
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        gen = torch.Generator().manual_seed(w.seed + 1000)
        go = torch.randn(w.B, w.H, 16384, w.d, generator=gen).bfloat16().to(dev)
        for _ in range(3):
            cl.backward(g["q"], g["k"], g["v"], go, g["a"], "elu1")
    elif case == "decode-small":
        w = W.DECODE
        B = 64                                       # B64 H32 d128: 128 MiB of state
        pre = W.decode_prefill_inputs(w, B=B)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in pre.items()}
        _, mu, nu = cl.forward_with_state(g["q"], g["k"], g["v"], g["a"], "elu1")
        for step in range(5):
            st = {k: v.to(dev) for k, v in W.decode_step_inputs(w, step, B=B).items()}
            cl.decode_step(mu, nu, st["q"], st["k"], st["v"], g["a"])
    else:
        raise SystemExit(f"unknown profile case {case}")
    torch.cuda.synchronize()
    status = cl.last_device_status()
    print(json.dumps({"profile_case": case, "device_status": status}))
    return 0 if status == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile-case", choices=["forward-long-small", "performer", "decode-small",
                                               "noncausal-long-small", "elu1-decay",
                                               "performer-decode-small", "token-decay-small",
                                               "backward-small", "backward-long-small"],
                    default=None,
                    help="run a small seeded case for an ncu capture and exit")
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args.profile_case)
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)
    dist = None
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = dist_mod
    try:
        return run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
