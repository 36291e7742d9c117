#!/usr/bin/env python
"""Benchmark of the tiered-KV decode hot path on GB300.

A step is one decode step of the whole attention stack over one batch: for
every layer, append the new token's K/V, fetch that layer's T1 rows (and, on
the first step after a re-tier, the delta of newly promoted rows) from pinned
host memory, run decode attention over T0/T1/T2 with the fused attention-weight
sums; then fold the scores; every Delta = 64 steps, re-tier.

Default workload: the 70B-shaped stack (80 layers, 64/8 heads, d 128, batch 8)
at the end of its 16,384-token sequences, T0 30 % / T1 67 % (pinned host) /
T3 3 %, the largest configuration that fits one GPU.  The timed steps contain a
re-tier step and the step after it (which carries the delta prefetch).  Inputs
are synthetic (seeded generator), already in HBM for `value`; `e2e` repeats the
timing with every step's q/k/v copied in from pinned host memory and the
outputs copied back inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 70b|32b|14b|7b|tiny]
                       [--impl tkv|reference] [--t0 R] [--t3 R] [--t1 ce|...] [--t2 hbm|host]
Under torchrun (N > 1) every rank runs its own replica (the path shards by
sequence, with no data-path collective); the timing is max over ranks.
"""
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

METRIC = "tiered decode-attn tokens/s (HBM GB/s vs peak); delta-prefetch PCIe GB/s"
# Decode steps before the profiled pass: two re-tiers (after steps 64 and 128).  The first
# only demotes (every token starts in T0); the second also promotes, so the profiled
# pass that follows it carries a delta prefetch.
PRE_STEPS = 128
TARGET_N = {"tiny": 640, "7b": 2512, "14b": 4096, "32b": 8192, "70b": 16384}
DESCR = {
    "tiny": "Tiny: 1 layer, 4/2 heads, d 64, batch 1",
    "7b": "7B-shaped attention stack: 28 layers, 28/4 heads, d 128, batch 1",
    "14b": "14B-shaped: 48 layers, 40/8 heads, d 128, batch 8",
    "32b": "32B-shaped: 64 layers, 40/8 heads, d 128, batch 4, T2 FP8-E4M3",
    "70b": "70B-shaped: 80 layers, 64/8 heads, d 128, batch 8",
}
LINK_PROBE_BYTES = 1 << 30
NOMINAL_PCIE5_X16_GBS = 64.0


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["tkv", "reference"], default="tkv")
    p.add_argument("--workload", default="70b", choices=sorted(TARGET_N))
    p.add_argument("--t0", type=float, default=None, help="T0 (HBM) ratio; T1 takes the rest")
    p.add_argument("--t3", type=float, default=None, help="eviction ratio")
    p.add_argument("--layers", type=int, default=None,
                   help="override the layer count (small captures for ncu; per-launch size unchanged)")
    p.add_argument("--t2", choices=["hbm", "host"], default="hbm",
                   help="where T2 (fp8) rows live: an HBM pool, or pinned host memory staged per layer")
    p.add_argument("--t1", choices=["ce", "sm", "split", "multi", "resident"], default="ce",
                   help="T1 transport: copy engine, SM copy kernel, both, four copy streams, or an "
                        "HBM-resident copy updated by the re-tier (only the delta crosses the link)")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-exposed", action="store_true",
                   help="skip the all-T0 run that measures the exposed transfer overhead")
    p.add_argument("--mode", choices=["graph", "eager"], default="graph",
                   help="timed steps: replays of a captured decode step, or eager per-layer calls")
    p.add_argument("--oracle-worker", action="store_true", help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ------------------------------------------------------------------ timeline
def prof_steps(steps):
    """Eager steps of the profiled pass that times every kernel and copy."""
    return max(4, min(steps, 16))


def timeline(steps, warmup, delta=64):
    """Decode-step numbers (from 1) of every phase of a run:
         1 .. PRE_STEPS             lead-in, re-tiers after steps 64 and 128;
         prof0 .. prof0 + kp - 1    profiled pass (eager; the first step carries the delta
                                    prefetch of the re-tier after step 128);
         fill0 .. warm0 - 1         filler (untimed);
         warm0 .. timed0 - 1        warm-up;
         timed0 .. last             the timed steps.
    With two or more timed steps the window is placed so that its middle holds a re-tier
    step (t % delta == 0) and the step after it (the delta prefetch)."""
    kp = prof_steps(steps)
    s_min = PRE_STEPS + kp + warmup + 1
    half = steps // 2
    if steps >= 2:
        r = delta * -(-(s_min + half - 1) // delta)
        s0 = r - half + 1
    else:
        s0 = s_min
    last = s0 + steps - 1
    return {"kp": kp, "prof0": PRE_STEPS + 1, "fill0": PRE_STEPS + kp + 1, "warm0": s0 - warmup,
            "timed0": s0, "last": last,
            "retiers_timed": [t for t in range(s0, last + 1) if t % delta == 0]}


def bench_workload(name, warmup, steps, t0=None, t3=None, layers=None):
    """The workload of a run: the configuration's shape and tiers, pre-filled so that the
    last timed step ends at the configuration's token count."""
    from tiered_kv_cache_gqa_gb300 import synth
    wl = synth.WORKLOADS[name]
    if layers:
        wl = wl.with_(num_layers=layers)
    r = list(wl.ratios)
    if t3 is not None:
        r[3] = t3
    if t0 is not None:
        r[0] = t0
    if t0 is not None or t3 is not None:
        r[1] = max(0.0, 1.0 - r[0] - r[2] - r[3])
    tl = timeline(steps, warmup, wl.delta)
    n_pre = max(wl.prompt_len + wl.window + 1, TARGET_N[name] - tl["last"])
    return wl.with_(ratios=tuple(r), prefill_len=n_pre, decode_steps=tl["last"])


def synth_layers(name):
    from tiered_kv_cache_gqa_gb300 import synth
    return synth.WORKLOADS[name].num_layers


def describe(wl):
    layers = "" if wl.num_layers == synth_layers(wl.name) else " [%d layers only]" % wl.num_layers
    return ("%s%s; %d pre-filled positions (prompt %d) + %d decode steps (re-tier every %d); "
            "tiers T0 %.0f%% T1 %.0f%% T2 %.0f%% T3 %.0f%%; sinks %d, window %d"
            % (DESCR[wl.name], layers, wl.prefill_len, wl.prompt_len, wl.decode_steps, wl.delta,
               *(100 * x for x in wl.ratios), wl.num_sinks, wl.window))


def kv_full_bytes(wl):
    """bf16 K/V bytes of every position at the end of the run (no tiering)."""
    return wl.num_layers * wl.batch * wl.max_tokens * 2 * wl.num_kv_heads * wl.head_dim * 2


def run_config(args, wl):
    """The `config` object of the JSON line; identical in both arms for the same arguments."""
    graph = args.mode == "graph" and args.t1 != "split"
    tl = timeline(args.steps, args.warmup, wl.delta)
    return {"workload": describe(wl), "inputs": "bf16 K/V/q (T2 rows FP8-E4M3)",
            "global_batch": wl.batch * args.gpus, "seq_len": TARGET_N[args.workload],
            "parallelism": "replicas (sequence shards)", "t1_transport": args.t1,
            "t2_placement": args.t2, "steps_as": "graph" if graph else "eager",
            "timed_steps": [tl["timed0"], tl["last"]], "retier_steps_timed": tl["retiers_timed"],
            "l2": "flushed between timed steps (256 MB write); full KV %.0f MB"
                  % (kv_full_bytes(wl) / 2 ** 20)}


def ncu_traffic_ratio(workload):
    """DRAM bytes (read + write) per attention launch over its algorithmic bytes, from the
    committed ncu summary of this workload's attention kernel, if it was captured from the
    attention source as it is now; else None.  The summary holds a line
    `traffic_ratio: <workload> <ratio> <sha256 of attention.cu>`."""
    import hashlib
    src = os.path.join(ROOT, "tiered_kv_cache_gqa_gb300", "csrc", "attention.cu")
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
        for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
            for line in open(os.path.join(ROOT, "profiles", name)):
                f = line.strip().strip("`").split()
                if len(f) == 4 and f[0] == "traffic_ratio:" and f[1] == workload and f[3] == digest:
                    return float(f[2])
    except OSError:
        return None
    return None


# ------------------------------------------------------------------ oracle arm
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def full_oracle_steps(wl):
    """Small stacks run whole oracle decode steps; large ones are sampled."""
    return wl.num_layers * wl.batch * wl.prefill_len <= 28 * 1 * 4096


def _oracle_pass_worker(wl, units, budget_s, seed_offset, queue):
    """One process: times single (sequence, layer) attention passes of the oracle over every
    position of the workload, until `budget_s` of timed work; K/V are drawn untimed."""
    import torch
    torch.set_num_threads(1)
    from oracle import attention
    from tiered_kv_cache_gqa_gb300 import synth
    gen = synth.Generator(wl, device="cpu")
    q_all, _, _ = gen.decode_step(1)
    done, t_total = 0, 0.0
    for (b, layer) in units:
        k, v = gen.kv_rows(b, layer, 0, wl.prefill_len)
        Kl = k.transpose(0, 1).double().numpy()
        Vl = v.transpose(0, 1).double().numpy()
        q = q_all[layer, b].double().numpy()
        t0 = time.perf_counter()
        attention.attend(q, Kl, Vl, wl.group)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total >= budget_s:
            break
    queue.put((done, t_total))


def oracle_run(wl, seconds, n_steps=0):
    """Times the fp64 oracle on this host.  Returns (tokens/s, description, cores used).

    Small stacks (Tiny, 7B) run whole decode steps of the oracle session, single-threaded
    (the session is sequential).  Larger ones are sampled: one worker process per host core
    times single (sequence, layer) attention passes over every position, and the step time
    is L * B passes at the workers' aggregate rate."""
    if full_oracle_steps(wl):
        os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        from oracle import session
        from tiered_kv_cache_gqa_gb300 import synth
        gen = synth.Generator(wl, device="cpu")
        sess = session.Session(wl.num_layers, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                               wl.batch, wl.prompt_len, wl.num_sinks, wl.window, wl.delta, wl.ratios)
        K, V = gen.prefill()
        sess.prefill(K.float().numpy(), V.float().numpy())
        done, t_total = 0, 0.0
        for t in range(1, wl.decode_steps + 1):
            q, k, v = gen.decode_step(t)
            a = (q.float().numpy(), k.float().numpy(), v.float().numpy())
            t0 = time.perf_counter()
            sess.step(*a)
            t_total += time.perf_counter() - t0
            done += 1
            if t_total >= seconds or (n_steps and done >= n_steps):
                break
        return wl.batch * done / t_total, "%d whole decode steps (all %d layers, batch %d), steps 1..%d" % (
            done, wl.num_layers, wl.batch, done), 1
    import multiprocessing as mp
    # one BLAS / OpenMP thread per worker process (inherited by the spawned children)
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cores = host_cores()
    workers = max(1, min(cores, 16))
    units = [(b, l) for l in range(wl.num_layers) for b in range(wl.batch)]
    per = [units[w::workers] for w in range(workers)]
    budget = max(1.0, 2.0 * seconds / workers)
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_oracle_pass_worker, args=(wl, per[w], budget, w, queue))
             for w in range(workers) if per[w]]
    for p in procs:
        p.start()
    res = [queue.get() for _ in procs]
    for p in procs:
        p.join()
    passes = sum(r[0] for r in res)
    rate = sum(r[0] / r[1] for r in res if r[1] > 0)          # passes per second, all workers
    step_s = wl.num_layers * wl.batch / rate
    return wl.batch / step_s, ("sampled: %d (sequence, layer) attention passes over %d positions on %d "
                               "worker processes (one per host core, single-threaded BLAS), step = "
                               "L*B = %d passes at their aggregate rate"
                               % (passes, wl.prefill_len, len(procs), wl.num_layers * wl.batch)), len(procs)


def oracle_worker(args):
    wl = bench_workload(args.workload, args.warmup, args.steps, args.t0, args.t3, args.layers)
    v, what, cores = oracle_run(wl, args.cpu_seconds)
    print(json.dumps({"value": v, "sample": what, "cores": cores}))


def cpu_baseline(args):
    """The oracle timed in a child process (no CUDA in it), before this process touches CUDA."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker", "--workload", args.workload,
           "--steps", str(args.steps), "--warmup", str(args.warmup),
           "--cpu-seconds", str(args.cpu_seconds)]
    if args.t0 is not None:
        cmd += ["--t0", str(args.t0)]
    if args.t3 is not None:
        cmd += ["--t3", str(args.t3)]
    if args.layers:
        cmd += ["--layers", str(args.layers)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle worker failed:\n" + r.stderr[-2000:])
    out = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": out["value"], "unit": "tokens/s", "cores": out["cores"],
            "host_cores": host_cores(), "kind": "oracle", "sample": out["sample"]}


# -------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) with their timestamps, written to a temporary file;
    `stop(t0, t1)` keeps the samples taken inside the wall-clock window [t0, t1]."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 100

    def __init__(self, index):
        self.index = index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="tkv_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def halt(self):
        if self.proc:
            time.sleep(0.3)          # let the sample after the window arrive
            self.proc.terminate()
            self.proc.wait()
            self.f.close()
            self.proc = None

    def read(self, t0=None, t1=None):
        import datetime
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            lines = open(self.path).readlines()
        except OSError:
            lines = []
        for line in lines:
            r = [x.strip() for x in line.split(",")]
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(r[2]), float(r[3])
            except (ValueError, IndexError):
                continue
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            sm.append(clk)
            mx = cmax
            for n, x in zip(names, r[6:10]):
                if x.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "window_s": (t1 - t0) if t0 is not None else None}

    def stop(self, t0=None, t1=None):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.halt()
        out = self.read(t0, t1)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        return out


def clocks_of(sampler, windows):
    """Clock record of the first window in `windows` [(label, t0, t1)] that holds at least
    three samples (a short timed window falls back to the loaded span around it)."""
    if not sampler or not sampler.proc:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    sampler.halt()
    out = None
    for label, t0, t1 in windows:
        out = sampler.read(t0, t1)
        out["window"] = label
        if out["samples"] >= 3:
            break
    try:
        os.unlink(sampler.path)
    except OSError:
        pass
    return out


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, rank, world):
    import numpy as np  # noqa: F401
    import torch
    import tiered_kv_cache_gqa_gb300 as tkv
    from tiered_kv_cache_gqa_gb300 import synth

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    tkv.load()
    wl = bench_workload(args.workload, args.warmup, args.steps, args.t0, args.t3, args.layers)
    wl = wl.with_(seed=rank_seed(wl.seed, rank))
    tl = timeline(args.steps, args.warmup, wl.delta)
    KP = tl["kp"]
    L, B, Hq, Hkv, d = wl.num_layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    stream = torch.cuda.current_stream()
    t1_mode = {"ce": tkv.TKV_T1_COPY_ENGINE, "sm": tkv.TKV_T1_SM_COPY, "split": tkv.TKV_T1_SPLIT,
               "multi": tkv.TKV_T1_MULTI_CE, "resident": tkv.TKV_T1_RESIDENT}[args.t1]
    # the split T1 transport is not capturable: its steps run eagerly
    graph = args.mode == "graph" and args.t1 != "split"
    t2_place = tkv.TKV_T2_HOST if args.t2 == "host" else tkv.TKV_T2_HBM

    def create(w, **kw):
        return tkv.TieredKV.for_workload(w, device=dev, t1_transport=t1_mode, t2_placement=t2_place, **kw)

    # The timed context's pinned host stores are allocated first, before this process frees
    # any host memory (the T1 stream reads them every step).
    ctx = create(wl)
    # the host link of this machine, measured in this run
    rc, link = tkv.tkv_measure_host_link(dev, LINK_PROBE_BYTES)
    if rc != tkv.TKV_OK:
        link = None
    else:
        link["bytes"] = LINK_PROBE_BYTES

    gen = synth.Generator(wl, device="cuda")
    n_steps = tl["last"]
    inputs = [gen.decode_step(t) for t in range(1, n_steps + 1)]
    # every context starts from the same pre-filled positions: drawn once, kept on the device
    prefill = [gen.prefill_layer(l) for l in range(L)]
    out = torch.empty(L, B, Hq, d, dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # > 129 MB L2
    # a captured step reads fixed buffers: each step's inputs are copied into them first
    sq, sk, sv = (torch.empty_like(x) for x in inputs[0])

    def fill(c, w):
        for l in range(L):
            c.append(l, prefill[l][0], prefill[l][1], w.prefill_len)
        return c

    class Stepper:
        """One decode step per call: eager per-layer calls, or a replay of a captured step
        (captured again whenever the last capture ran out or a re-tier discarded it)."""

        def __init__(self, c):
            self.c, self.left, self.captures, self.retiers = c, 0, 0, 0

        def eager(self, t, q, k, v):
            for l in range(L):
                self.c.append(l, k[l], v[l], 1)
                if l == 0:
                    self.c.prefetch(0)
                if l + 1 < L:
                    self.c.prefetch(l + 1)
                self.c.decode_step(l, q[l], out[l])

        def __call__(self, t, q, k, v, use_graph):
            if use_graph:
                sq.copy_(q, non_blocking=True)
                sk.copy_(k, non_blocking=True)
                sv.copy_(v, non_blocking=True)
                # the step after a re-tier carries the delta prefetch: eager
                if self.left == 0 and (t - 1) % wl.delta != 0:
                    self.c.capture_begin()
                    self.eager(t, sq, sk, sv)
                    self.left = self.c.capture_end()
                    self.captures += 1
                if self.left > 0:
                    self.c.replay()
                    self.left -= 1
                else:
                    self.eager(t, sq, sk, sv)
            else:
                self.eager(t, q, k, v)
            if t % wl.delta == 0:
                self.c.retier()
                self.retiers += 1
                self.left = 0

    def lead_in(c, r, profile):
        """Steps 1 .. timed0 - 1 (see `timeline`); returns the profiled pass."""
        for t in range(1, tl["prof0"]):
            r(t, *inputs[t - 1], False)
        prof = None
        if profile:
            c.profile_begin()
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(KP)]
        for i, t in enumerate(range(tl["prof0"], tl["fill0"])):
            flush.fill_(i & 0xFF)
            pev[i][0].record(stream)
            r(t, *inputs[t - 1], False)
            pev[i][1].record(stream)
        if profile:
            prof = c.profile_end()
        torch.cuda.synchronize()
        prof_ms = sum(x.elapsed_time(y) for x, y in pev)
        for t in range(tl["fill0"], tl["timed0"]):
            r(t, *inputs[t - 1], graph)
        c.sync()
        torch.cuda.synchronize()
        return prof, prof_ms

    def timed(c, r):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        launches0 = c.stats()["kernel_launches"]
        captures0, retiers0 = r.captures, r.retiers
        # marks the timed region for a profiler started with collection off (no-op otherwise)
        torch.cuda.profiler.start()
        for i, t in enumerate(range(tl["timed0"], tl["last"] + 1)):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            r(t, *inputs[t - 1], graph)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        w1 = time.time()
        torch.cuda.profiler.stop()
        if world > 1:
            torch.distributed.barrier()
        step_ms = [x.elapsed_time(y) for x, y in ev]
        return {"step_ms": step_ms, "w0": w0, "w1": w1,
                "launches": c.stats()["kernel_launches"] - launches0,
                "captures": r.captures - captures0, "retiers": r.retiers - retiers0}

    # clocks: sampled from before the lead-in; the samples inside the timed window are kept
    sampler = ClockSampler(dev) if rank == 0 else None
    if sampler:
        sampler.start()
    fill(ctx, wl)
    run = Stepper(ctx)
    wl0 = time.time()
    prof, prof_ms = lead_in(ctx, run, True)
    tm = timed(ctx, run)
    clocks = clocks_of(sampler, [("timed", tm["w0"], tm["w1"]), ("filler + warm-up + timed", wl0, tm["w1"])])
    total_ms = sum(tm["step_ms"])
    st = ctx.stats()
    ctx.close()

    # ---- exposed transfer overhead: the same timeline with every retained row in T0
    exposed = None
    if not args.no_exposed:
        r3 = wl.ratios[3]
        wl_t0 = wl.with_(ratios=(1.0 - r3, 0.0, 0.0, r3))
        c0 = fill(create(wl_t0, t1_capacity=256, t2_capacity=1), wl_t0)   # small host stores: T1 holds a rounding remainder at most
        r0 = Stepper(c0)
        lead_in(c0, r0, False)
        tm0 = timed(c0, r0)
        c0.close()
        exposed = {"all_t0_ms_per_step": sum(tm0["step_ms"]) / args.steps,
                   "share": (total_ms - sum(tm0["step_ms"])) / total_ms}

    # ---- e2e: the same steps fed from pinned host buffers, outputs copied back
    e2e = None
    if not args.no_e2e:
        steps_in = inputs[tl["timed0"] - 1: tl["last"]]
        host_in = [(q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()) for (q, k, v) in steps_in]
        dq, dk, dv = (torch.empty_like(x) for x in inputs[0])
        host_out = torch.empty(L, B, Hq, d, dtype=torch.float32).pin_memory()
        # the same decode positions on a fresh context, so both loops see the same state
        ctx = fill(create(wl), wl)
        run = Stepper(ctx)
        lead_in(ctx, run, False)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for i, t in enumerate(range(tl["timed0"], tl["last"] + 1)):
            qh, kh, vh = host_in[i]
            dq.copy_(qh, non_blocking=True)
            dk.copy_(kh, non_blocking=True)
            dv.copy_(vh, non_blocking=True)
            run(t, dq, dk, dv, graph)
            host_out.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        h2d = sum(x.numel() * x.element_size() for x in host_in[0])
        d2h = host_out.numel() * host_out.element_size()
        e2e = {"ms": e2e_ms, "h2d": h2d, "d2h": d2h}
        ctx.close()
    return {"total_ms": total_ms, "tm": tm, "prof": prof, "stats": st, "clocks": clocks, "wl": wl,
            "e2e": e2e, "prof_steps": KP, "prof_ms": prof_ms, "exposed": exposed, "link": link}


# ------------------------------------------------------------------ ranks
# Replicas: every rank runs its own sequences (weak scaling, no data-path collective); only the
# timing crosses ranks.
def rank_seed(seed, rank):
    """Seed of a rank's sequences: distinct sequences per rank."""
    return seed + 1000 * rank


def max_over_ranks(values):
    """Element-wise max of a list of floats over every rank (gloo all-reduce); the input when
    there is one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_tokens_per_s(batch, steps, world, max_ms):
    """Tokens decoded by all ranks over the slowest rank's time."""
    return batch * steps * world / (max_ms / 1e3)


def hbm_projection(wl, args):
    """HBM saved by tiering at the end of the run, from the footprint calculator at the
    workload's shape, batch, token count and tier ratios (steady state)."""
    from tiered_kv_cache_gqa_gb300 import memory
    f = memory.projection(wl.num_layers, wl.batch, wl.num_kv_heads, wl.head_dim, wl.max_tokens,
                          wl.ratios, prompt_len=wl.prompt_len, num_sinks=wl.num_sinks, window=wl.window,
                          t1_resident=args.t1 == "resident", t2_on_host=args.t2 == "host")
    return f.saved_bytes


def link_bound_step_ms(t1_bytes_per_step, link):
    """Time a step's T1 rows take at the measured copy-engine link peak (ms), or None."""
    if not link or not link.get("h2d_ce_gbs") or t1_bytes_per_step <= 0:
        return None
    return t1_bytes_per_step / (link["h2d_ce_gbs"] * 1e9) * 1e3


def link_fraction(gbs, link):
    """A host-link rate as fractions of the measured link peak and of nominal PCIe Gen5 x16."""
    if gbs is None:
        return None
    peak = max(link["h2d_ce_gbs"], link["h2d_sm_gbs"]) if link else None
    return {"gbs": gbs, "frac_of_measured_link": (gbs / peak) if peak else None,
            "frac_of_nominal_pcie5x16": gbs / NOMINAL_PCIE5_X16_GBS}


def main():
    args = parse()
    if args.oracle_worker:
        oracle_worker(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    wl = bench_workload(args.workload, args.warmup, args.steps, args.t0, args.t3, args.layers)

    if args.impl == "reference":
        # the oracle on this host's cores, on the same workload; other ranks do nothing
        if rank == 0:
            v, what, cores = oracle_run(wl, args.cpu_seconds)
            line = {"metric": METRIC, "impl": "reference", "value": v, "unit": "tokens/s",
                    "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": 1000.0 * wl.batch / v, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                    "config": run_config(args, wl),
                    "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores,
                                     "host_cores": host_cores(), "kind": "oracle", "sample": what},
                    "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    r = run_gpu(args, rank, world)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # a child process with no GPU (its oracle workers are spawned, not forked)
        cpu = cpu_baseline(args)
    total_ms = r["total_ms"]
    e2e_ms = r["e2e"]["ms"] if r["e2e"] else None
    m = max_over_ranks([total_ms, e2e_ms or 0.0])
    total_ms, e2e_ms = m[0], (m[1] if e2e_ms is not None else None)
    if rank != 0:
        return
    wl = r["wl"]
    K = args.steps
    tokens = wl.batch * K * world
    value = whole_job_tokens_per_s(wl.batch, K, world, total_ms)
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        hbm_peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except Exception:
        hbm_peak, peak_src = 6800.0, "fallback"
    pa, pc, p1, pd = r["prof"]["attn"], r["prof"]["combine"], r["prof"]["t1"], r["prof"]["delta"]
    KP_ = r["prof_steps"]
    # DRAM bytes per launch: the ncu-measured ratio to the algorithmic bytes, scaled to this
    # run's launches (traffic grows with the retained rows a launch reads)
    ratio = ncu_traffic_ratio(args.workload) if not args.layers else None
    traffic = ratio * pa["bytes"] / max(1, pa["count"]) if ratio else None
    achieved = pa["bytes"] / (pa["ms"] / 1e3) / 1e9 if pa["ms"] > 0 else 0.0
    st = r["stats"]
    tm = r["tm"]
    t1_gbs = p1["bytes"] / (p1["ms"] / 1e3) / 1e9 if p1["ms"] > 0 else None
    delta_gbs = pd["bytes"] / (pd["ms"] / 1e3) / 1e9 if pd["ms"] > 0 else None
    link_ms = p1["ms"] + pd["ms"]
    tl = timeline(args.steps, args.warmup, wl.delta)
    link_floor = link_bound_step_ms(p1["bytes"] / KP_ if KP_ else 0.0, r["link"])
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": run_config(args, wl),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "kernel": "tkv::attn_kernel", "peak_source": peak_src,
                     "launches": pa["count"], "avg_launch_us": 1e3 * pa["ms"] / max(1, pa["count"]),
                     "bytes_per_launch": pa["bytes"] / max(1, pa["count"]),
                     "note": "main attention kernel alone (CUDA events on the compute stream, eager "
                             "profiled steps); the combine kernel that follows it is in detail.attention_combine"},
        "cpu_baseline": cpu,
        "e2e": ({"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                 "h2d_bytes_per_step": r["e2e"]["h2d"], "d2h_bytes_per_step": r["e2e"]["d2h"]}
                if e2e_ms else None),
        "gpu_launches": tm["launches"],
        "clocks": r["clocks"],
        "detail": {
            "timed_region": {"captures": tm["captures"], "retiers": tm["retiers"],
                             "step_ms": [round(x, 3) for x in tm["step_ms"]],
                             "steps": [tl["timed0"], tl["last"]]},
            "profiled_pass": {"steps": KP_, "first_step": tl["prof0"], "mode": "eager",
                              "ms_per_step": r["prof_ms"] / KP_,
                              "note": "per-kernel events; roofline and transfer figures come from this pass"},
            "attention_step_ms": (pa["ms"] + pc["ms"]) / KP_,
            "attention_combine": {"avg_launch_us": 1e3 * pc["ms"] / max(1, pc["count"]),
                                  "launches": pc["count"], "bytes_per_launch": pc["bytes"] / max(1, pc["count"]),
                                  "pair_frac_of_hbm_peak": ((pa["bytes"] + pc["bytes"]) / ((pa["ms"] + pc["ms"]) / 1e3)
                                                            / 1e9 / hbm_peak) if pa["ms"] + pc["ms"] > 0 else None},
            "host_link_measured": r["link"],
            "host_stores": {"bytes": st["host_bytes_allocated"], "huge_page_bytes": st["host_huge_bytes"],
                            "numa_node": st["host_numa_node"]},
            "t1_stream": dict(link_fraction(t1_gbs, r["link"]) or {}, bytes_per_step=p1["bytes"] / KP_,
                              ms_per_step=p1["ms"] / KP_, t2_bytes_total=st["h2d_bytes_t2_stream"],
                              note="host-link stream per layer: T1 rows, and T2 records with --t2 host"),
            "delta_prefetch": dict(link_fraction(delta_gbs, r["link"]) or {}, bytes=pd["bytes"], ms=pd["ms"],
                                   launches=pd["count"]),
            "transfer_overhead_copy_share": link_ms / r["prof_ms"],
            "transfer_overhead_exposed": r["exposed"],
            "hbm_saved_bytes": st["kv_bytes_full_cache"] - st["hbm_bytes_kv_resident"],
            "hbm_saved_projection_bytes": hbm_projection(wl, args),
            "hbm_kv_resident_bytes": st["hbm_bytes_kv_resident"],
            "kv_full_cache_bytes": st["kv_bytes_full_cache"],
            "tier_count": st["tier_count"],
            "step_ms_median": statistics.median(tm["step_ms"]),
            "host_link_floor": link_floor and {
                "ms_per_step": link_floor,
                "timed_steps_within_10pct": sum(1 for x in tm["step_ms"] if x <= 1.1 * link_floor),
                "note": "a step's T1 bytes at the link peak measured in this run: no step can be faster "
                        "while T1 crosses the link every step; slower steps read the host store slower"},
        },
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
