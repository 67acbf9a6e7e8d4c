#!/usr/bin/env python3
"""Benchmark of the fused rank-sum + residual add + RMSNorm operator.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl farn|reference]

One step is one pass of the whole operator over one batch of the workload:
for the default workload, the largest benchmark configuration (W=4,
T=32768, H=5120: 2.68 GB per call), one call on the full [T,H] problem; for
the decode sweep (W=8, H=4096), one call for each T in 1,2,4,...,128 (255
rows).  The headline workload runs exactly --steps timed steps; then every
other benchmark configuration (c1, decode, prefill, nonpow2, wide) is timed
in the same run and reported under "configs" (--only skips them).  Inputs are seeded synthetic bf16 tensors generated on the
device (synth/), rotated over enough copies that one pass over all copies
is more than twice the L2 cache, so every call reads HBM.

Metric: effective bytes per second, counting (W+1)*T*H*2 bytes read, H*2
bytes of weight and 3*T*H*2 bytes written per call, and rows per second,
as a fraction of the measured HBM copy bandwidth; next to the CPU oracle
timed on the host's cores.  `value` is the device-timed throughput with
inputs resident in HBM (CUDA events around K graph replays); `e2e` times
the same calls with the inputs copied from pinned host memory and the
outputs copied back inside the timed region.

--impl reference times the CPU oracle (the only other implementation of
this operator; there is no upstream package to install) on bounded samples
of the same workload.

Multi-GPU: one process per GPU (torchrun); the operator has no exchange
step, so each rank runs its own replica (weak scaling); the time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s and rows/s (1×GB300) as % of HBM peak, vs CPU oracle"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "nonpow2"
# The benchmark configurations: a small call, the decode sweep, prefill, a
# non-power-of-two hidden size and a wide reduction.
BENCH_CONFIGS = ("c1", "decode", "prefill", "nonpow2", "wide")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 1.5 s of GPU time)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["decode", "c1", "prefill", "nonpow2", "wide", "rmsnorm",
                             "prefill_f32", "prefill_fp8", "prefill_nvfp4", "moe_combine"])
    ap.add_argument("--in-place", action="store_true",
                    help="write residual_out over the residual (in-place residual update)")
    ap.add_argument("--impl", default="farn", choices=["farn", "reference"])
    ap.add_argument("--no-graph", action="store_true",
                    help="launch each call from Python instead of replaying a CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU oracle work for cpu_baseline (rank 0)")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="--impl reference: oracle time budget for the whole run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--rows", type=int, default=None,
                    help="override T of every call (small cases for profiling)")
    ap.add_argument("--only", action="store_true",
                    help="time the --workload alone, not the other benchmark configurations")
    ap.add_argument("--config-ms", type=float, default=300.0,
                    help="timed GPU work per extra configuration, ms")
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0,
                    help="CPU oracle work per extra configuration")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- helpers
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks (the slowest rank's time); the
    identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_info():
    model = platform.processor() or ""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu part", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"machine": platform.machine(), "nproc": os.cpu_count(), "cpu": model}


class ClockSampler:
    """nvidia-smi samples (host wall time, SM MHz, max MHz, reasons)."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str | None):
        self.samples, self.proc, self.thread = [], None, None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            reasons = [n for n, v in zip(self.NAMES, parts[3:]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, smax, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "samples inside the timed region"
        if not inside and self.samples:
            # region shorter than the sampling period: nearest samples
            mid = 0.5 * (t0 + t1)
            inside = sorted(self.samples, key=lambda s: abs(s[0] - mid))[:3]
            note = "timed region shorter than the sampling period; nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "nvidia-smi unavailable"}
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "note": note}


def gpu_id_for(dev_index):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# -------------------------------------------------------- CPU (the oracle)
def row_bytes(p) -> int:
    """Algorithmic bytes of one row of a call (weight counted per call)."""
    return (p.algorithmic_bytes() - p.H * 2) // p.T


def call_bytes(p, rows) -> int:
    return rows * row_bytes(p) + p.H * 2


def oracle_sampler(problems, seed_rows=8):
    """Host copies of a few rows per problem, made with the numpy twin of
    the generator (the oracle's own input path), for CPU timing."""
    import synth
    out = []
    for p in problems:
        rows = min(p.T, seed_rows)
        xs, res, w = synth.host_inputs(p.with_T(rows))
        out.append((p, xs, res, w))
    return out


def time_oracle_rows(sample, rows_total_target=None, seconds=10.0):
    """Run the oracle over the sample's rows repeatedly for about `seconds`.
    Returns (bytes, rows, elapsed_s)."""
    import oracle
    O = oracle.Oracle()
    nbytes = nrows = 0
    t0 = time.perf_counter()
    while True:
        for p, xs, res, w in sample:
            if p.kind == "moe_combine":
                outs = O.moe_combine(*xs, res, w, p.eps)
            else:
                outs = O.forward(xs, res, w, p.eps)
            if p.fp8_out:
                O.quant_e4m3(outs[2])
            if p.nvfp4_out:
                O.quant_nvfp4(outs[2], p.tensor_scale)
            r = res.shape[0]
            nbytes += call_bytes(p, r)
            nrows += r
        el = time.perf_counter() - t0
        if el >= seconds:
            return nbytes, nrows, el


def cpu_baseline(problems, seconds):
    sample = oracle_sampler(problems)
    nbytes, nrows, el = time_oracle_rows(sample, seconds=seconds)
    desc = "; ".join(f"{p.name}: {min(p.T, 8)} rows" for p in problems)
    return {"value": nbytes / el / 1e9, "unit": UNIT, "rows_per_s": nrows / el,
            "cores": 1, "kind": "oracle",
            "sample": f"single-threaded C oracle, repeated for {el:.1f} s over "
                      f"seeded rows of the same shapes ({desc})",
            **host_info()}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    import synth
    problems = synth.workload(args.workload)
    K = args.steps if args.steps is not None else 30
    Wu = args.warmup
    sample = oracle_sampler(problems)
    # calibrate: seconds per row
    nb, nr, el = time_oracle_rows(sample, seconds=0.5)
    s_per_row = el / max(nr, 1)
    rows_per_step = max(1, int(args.reference_seconds / (K + Wu) / s_per_row))
    import oracle
    O = oracle.Oracle()
    cursor = 0

    def step():
        """At least rows_per_step rows: whole sampled blocks (up to 8 rows of
        one call each), handed to the oracle as they are."""
        nonlocal cursor
        b = n = 0
        while n < rows_per_step:
            p, xs, res, w = sample[cursor % len(sample)]
            cursor += 1
            if p.kind == "moe_combine":
                outs = O.moe_combine(*xs, res, w, p.eps)
            else:
                outs = O.forward(xs, res, w, p.eps)
            if p.fp8_out:
                O.quant_e4m3(outs[2])
            if p.nvfp4_out:
                O.quant_nvfp4(outs[2], p.tensor_scale)
            r = res.shape[0]
            b += call_bytes(p, r)
            n += r
        return b, n

    for _ in range(Wu):
        step()
    tb = tn = 0
    t0 = time.perf_counter()
    for _ in range(K):
        b, n = step()
        tb += b
        tn += n
    el = time.perf_counter() - t0
    value = tb / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": K, "warmup": Wu,
        "ms_per_step": el / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "rows_per_s": tn / el,
        "config": {"workload": workload_desc(args.workload, problems),
                   "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1,
                         "kind": "oracle",
                         "sample": f"at least {rows_per_step} rows per step, in the "
                                   f"sampled blocks of up to 8 rows of each of the "
                                   f"workload's calls, one oracle call per block",
                         **host_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_desc(name, problems):
    p = problems[0]
    if name == "decode":
        return (f"decode sweep: W={p.W}, H={p.H}, T in "
                f"{{{','.join(str(q.T) for q in problems)}}} (one call per T), eps={p.eps:g}")
    out = ""
    if p.fp8_out:
        out = ", norm_out written as E4M3 + fp32 row scales (no bf16 norm_out)"
    elif p.nvfp4_out:
        out = (", norm_out written as NVFP4: E2M1 codes + E4M3 scales per 16 elements, "
               f"tensor scale {p.tensor_scale:g} (no bf16 norm_out)")
    if p.kind == "moe_combine":
        out = (f", MoE combine of K={p.W} gathered expert rows per token "
               "(seeded permutation, softmax gates)")
    return (f"{name}: W={p.W}, T={p.T}, H={p.H}, x ~ {p.x.describe()}, "
            f"residual ~ {p.residual.describe()}, weight ~ {p.weight.describe()}, eps={p.eps:g}"
            + out)


# ------------------------------------------------------------------ GPU
def setup_sets(problems, dev, stream, l2, in_place):
    """Rotating device copies of one workload's inputs and outputs, enough
    that one pass over all of them is more than twice the L2 size."""
    import torch
    import synth
    set_bytes = sum(p.algorithmic_bytes() for p in problems)
    n_sets = max(2, math.ceil(2 * l2 / set_bytes))
    n_sets = min(n_sets, max(1, int(40e9 // set_bytes)))
    sets = []
    with torch.cuda.stream(stream):
        for k in range(n_sets):
            calls = []
            for p in problems:
                xs, res, w = synth.device_inputs(p, dev, seed=p.seed + 7919 * k)
                outs = make_outputs(p, dev)
                if in_place:
                    # residual_out is the residual buffer itself; every step
                    # then reads the residual the previous step over that
                    # copy wrote, which leaves the bytes moved unchanged
                    outs = (outs[0], res) + tuple(outs[2:])
                calls.append((p, xs, res, w, outs))
            sets.append(calls)
    stream.synchronize()
    return sets, set_bytes


class StepRunner:
    """Steps of one workload over its rotating input copies.  One CUDA graph
    replay covers whole rotations, at least `min_block` steps (block steps),
    plus a one-step graph per copy, so exactly the requested number of
    steps is run, the host never paces the GPU, and few replay boundaries
    fall inside a short timed region."""

    def __init__(self, sets, ctx, stream, use_graph, min_block=10):
        import torch
        self.sets, self.ctx, self.stream = sets, ctx, stream
        self.n_sets = len(sets)
        self.block = self.n_sets * max(1, -(-min_block // self.n_sets))
        self.use_graph = use_graph
        self.graph, self.step_graphs, self.pos = None, [], 0
        if use_graph:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                for k in range(self.block):
                    self.step(k % self.n_sets)
            for k in range(self.n_sets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    self.step(k)
                self.step_graphs.append(g)
            self.graph.replay()
            for g in self.step_graphs:
                g.replay()
            stream.synchronize()

    def step(self, k):
        for p, xs, res, w, outs in self.sets[k]:
            call_forward(p, xs, res, w, outs, self.ctx, self.stream)

    def run(self, n):
        """Exactly n steps, continuing the rotation over the input copies."""
        while n > 0:
            if self.use_graph and self.pos == 0 and n >= self.block:
                self.graph.replay()
                n -= self.block
                continue
            if self.use_graph:
                self.step_graphs[self.pos].replay()
            else:
                self.step(self.pos)
            self.pos = (self.pos + 1) % self.n_sets
            n -= 1


def time_steps(runner, stream, dev, K, warmup, world, target_ms=1500.0):
    """Warm-up, then exactly K steps (K None: about target_ms of GPU time)
    timed with CUDA events on the launching stream, bracketed by a barrier
    and a device synchronisation; the time is the maximum over ranks."""
    import torch
    n_sets = runner.n_sets
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    runner.run(max(warmup, 1))
    stream.synchronize()
    e0.record(stream)
    runner.run(4 * n_sets)
    e1.record(stream)
    e1.synchronize()
    calib_ms = e0.elapsed_time(e1) / (4 * n_sets)
    if K is None:
        K = max(20, int(target_ms / max(calib_ms, 1e-4)))
        K = (K + n_sets - 1) // n_sets * n_sets
    runner.run(warmup)
    if runner.pos:
        # untimed steps up to the next whole rotation, so that the timed
        # steps start on a block graph
        runner.run(runner.n_sets - runner.pos)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    # The K steps run back to back; events between consecutive chunks of
    # them (recorded on the same stream, no gap added) give the spread.
    # Chunks are whole graph blocks where K allows, so that short timed
    # regions do not replay one-step graphs.
    n_chunks = max(1, min(20, K // runner.block if K >= runner.block else 1))
    bounds = [round(K * i / n_chunks) for i in range(n_chunks + 1)]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_chunks + 1)]
    t_wall0 = time.time()
    evs[0].record(stream)
    for i in range(n_chunks):
        runner.run(bounds[i + 1] - bounds[i])
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(evs[0].elapsed_time(evs[-1]), dev)
    chunk_ms = sorted(evs[i].elapsed_time(evs[i + 1]) / (bounds[i + 1] - bounds[i])
                      for i in range(n_chunks) if bounds[i + 1] > bounds[i])

    def pct(q):
        return chunk_ms[min(len(chunk_ms) - 1, int(q * (len(chunk_ms) - 1) + 0.5))]
    stats = {"chunks": len(chunk_ms), "p10_ms": pct(0.1), "median_ms": pct(0.5),
             "p90_ms": pct(0.9), "mean_ms": ms / K}
    return K, ms, stats, calib_ms, (t_wall0, t_wall1)


def annotate_calls(per_call, problems, sets, ctx, peak):
    """Per-call GB/s, fraction of the peak and the kernel plan."""
    import rank_sum_residual_gb300 as farn
    for j, c in enumerate(per_call):
        c["gbs"] = c["bytes"] / (c["kernel_us"] * 1e-6) / 1e9
        c["frac"] = c["gbs"] / peak
        c["rows_per_s"] = c["T"] / (c["kernel_us"] * 1e-6)
        if problems[j].kind == "moe_combine":
            _, (ex, _, _), res_j, w_j, outs_j = sets[0][j]
            v, thr = farn.farn_plan_moe_combine(
                ctx.handle, problems[j].W, problems[j].T, problems[j].H, ex.data_ptr(),
                res_j.data_ptr(), w_j.data_ptr(), outs_j[0].data_ptr(), outs_j[1].data_ptr(),
                outs_j[2].data_ptr())
            c["variant"] = ("combine-stage" if v == "stage" else v) + f" threads={thr}"
            continue
        v, cs, thr = farn.farn_plan_typed(ctx.handle, *plan_args(sets[0][j]))
        c["variant"] = f"{v} cluster={cs} threads={thr}"
        c["kernel"] = kernel_name(c["variant"])


# The acceptance bars on the fraction of the HBM roofline: long calls
# (T >= 4096) at least 75 %, decode-sized calls (T <= 128) at least 40 %.
def bar_for(T):
    return 0.75 if T >= 4096 else (0.40 if T <= 128 else None)


def config_summary(name, problems, K, ms, stats, calib_ms, per_call, n_sets, set_bytes, l2,
                   peak, world, clocks):
    step_bytes = sum(p.algorithmic_bytes() for p in problems)
    step_rows = sum(p.T for p in problems)
    secs = ms / 1e3
    gbs = world * step_bytes * K / secs / 1e9
    out = {"workload": workload_desc(name, problems), "steps": K, "ms_per_step": ms / K,
           "bytes_per_step": step_bytes, "rows_per_step": step_rows,
           "gbs": gbs, "frac": gbs / world / peak, "rows_per_s": world * step_rows * K / secs,
           "step_ms_spread": stats, "calibration_ms_per_step": calib_ms,
           "l2": f"inputs rotated over {n_sets} device copies "
                 f"({n_sets * set_bytes / 1e6:.0f} MB > 2 x L2 {l2 / 1e6:.0f} MB); no flush",
           "clocks": clocks,
           "per_call": per_call}
    bars = [(c["call"], bar_for(c["T"]), c["frac"]) for c in per_call if bar_for(c["T"])]
    if bars:
        out["bar"] = {c: {"target_frac": b, "frac": f, "met": f >= b} for c, b, f in bars}
    return out


def run_gpu(args):
    import torch

    import rank_sum_residual_gb300 as farn
    import synth
    from rank_sum_residual_gb300 import _build

    rank, world, local = dist_info()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build_library()
    synth.build()

    peak, peak_src = hbm_peak()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ctx = farn.Context(local)
    # One stream for everything: torch's graph replay, the calls and every
    # CUDA event all use torch's current stream, so make it this one.
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    use_graph = not args.no_graph

    def load(name):
        problems = synth.workload(name)
        if args.rows is not None:
            problems = [p.with_T(args.rows) for p in problems]
        return problems

    sampler = ClockSampler(gpu_id_for(local)).start() if rank == 0 else None
    time.sleep(0.5 if sampler else 0)

    # ---- the headline workload: exactly --steps timed steps after --warmup
    problems = load(args.workload)
    step_bytes = sum(p.algorithmic_bytes() for p in problems)
    step_rows = sum(p.T for p in problems)
    sets, set_bytes = setup_sets(problems, dev, stream, l2, args.in_place)
    runner = StepRunner(sets, ctx, stream, use_graph)
    K, ms, step_stats, calib_ms, (t_wall0, t_wall1) = time_steps(
        runner, stream, dev, args.steps, args.warmup, world)
    # per-call kernel time, right after the timed steps and under the same
    # clock sampling: each call alone, back to back over its own input copies
    per_call = time_calls_alone(problems, dev, ctx, l2)
    annotate_calls(per_call, problems, sets, ctx, peak)
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None

    secs = ms / 1e3
    value = world * step_bytes * K / secs / 1e9
    rows_per_s = world * step_rows * K / secs
    dom = max(per_call, key=lambda c: c["kernel_us"] * c["count_per_step"])
    roofline = {"bound": "hbm", "achieved": dom["gbs"], "peak": peak, "unit": "GB/s",
                "frac": dom["frac"], "traffic": measured_traffic(dom["call"], dom["variant"]),
                "kernel_source_sha": kernel_source_sha(),
                "kernel": kernel_name(dom["variant"]), "plan": dom["variant"],
                "call": dom["call"],
                "algorithmic_bytes_per_launch": dom["bytes"],
                "launch_us": dom["kernel_us"], "launches_timed": dom["launches_timed"],
                "peak_source": "measured: MEASURED_PEAKS.json hbm_gbs (copy bandwidth)"
                if peak_src == "measured" else "fallback 6.8 TB/s",
                "timing": "CUDA events around a graph of back-to-back launches of this "
                          "call alone over its own rotating copies (> 2 x L2), right "
                          "after the timed steps"}
    n_sets, block = runner.n_sets, runner.block
    head = config_summary(args.workload, problems, K, ms, step_stats, calib_ms, per_call,
                          n_sets, set_bytes, l2, peak, world, clocks)

    # ---- end to end: pinned host inputs in, outputs back, every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(sets[0], problems, stream, dev, K, world, step_bytes)
    del runner, sets
    torch.cuda.empty_cache()

    cpu = cpu_baseline(problems, args.cpu_seconds) if (rank == 0 and world == 1) else None
    head["cpu_baseline"] = cpu

    # ---- every other benchmark configuration, in the same run
    configs = {args.workload: head}
    others = [] if args.only else [n for n in BENCH_CONFIGS if n != args.workload]
    for name in others:
        probs = load(name)
        csets, cbytes = setup_sets(probs, dev, stream, l2, False)
        crun = StepRunner(csets, ctx, stream, use_graph)
        cK, cms, cstats, ccal, (c0, c1) = time_steps(
            crun, stream, dev, None, max(3, args.warmup), world, target_ms=args.config_ms)
        cper = time_calls_alone(probs, dev, ctx, l2)
        annotate_calls(cper, probs, csets, ctx, peak)
        cclk = sampler.summary(c0, c1) if sampler else None
        summ = config_summary(name, probs, cK, cms, cstats, ccal, cper, crun.n_sets, cbytes,
                              l2, peak, world, cclk)
        summ["cpu_baseline"] = (cpu_baseline(probs, args.config_cpu_seconds)
                                if (rank == 0 and world == 1) else None)
        configs[name] = summ
        del crun, csets
        torch.cuda.empty_cache()
    time.sleep(0.3 if sampler else 0)
    if sampler:
        sampler.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(args.workload, problems),
                       "calls_per_step": len(problems), "rows_per_step": step_rows,
                       "bytes_per_step": step_bytes,
                       "accumulate": "f32",
                       "residual_out": "in place over residual" if args.in_place else "separate",
                       "l2": head["l2"],
                       "launch": (f"CUDA graphs: one replay per {block} steps (whole "
                                  f"rotations of {n_sets} input copies), one-step graphs "
                                  "for the rest" if use_graph else "direct launches"),
                       "calibration_ms_per_step": calib_ms,
                       "timing": (f"exactly {K} back-to-back steps after {args.warmup} "
                                  "warm-up steps, CUDA events on the launching stream; "
                                  "the spread over chunks of them is step_ms_spread; "
                                  f"roofline.launch_us from {roofline['launches_timed']} "
                                  "launches of the call alone"),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "rows_per_s": rows_per_s,
            "pct_hbm_peak": 100.0 * value / world / peak,
            "step_ms_spread": step_stats,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": K * len(problems),
            "clocks": clocks,
            "per_call": per_call,
            "configs": configs,
            "configs_note": ("every benchmark configuration measured in this run: the "
                             "headline one with exactly --steps timed steps; each other one "
                             f"with about {args.config_ms:g} ms of timed steps, then each "
                             "call alone (per_call); each with its own oracle sample"),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


KERNELS = {"row": "farn_vec_kernel", "cluster": "farn_vec_kernel",
           "generic": "farn_generic_kernel", "bulk": "farn_bulk_kernel",
           "stage": "farn_stage_kernel", "combine": "farn_combine_kernel",
           "combine-stage": "farn_combine_stage_kernel"}
KERNEL_SOURCES = ("rank_sum_residual_gb300/csrc/farn_kernels.cuh",)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.md")


def kernel_name(variant):
    return KERNELS[variant.split()[0]]


def kernel_source_sha() -> str:
    """Hash of the kernel source: ncu counters taken with another hash
    describe another kernel."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(call: str, variant: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    of this call from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as fh:
            lines = fh.read().splitlines()
    except OSError:
        return None
    sha = kernel_source_sha()
    key = variant.replace(" ", "_")
    for line in lines:
        if not line.startswith("traffic "):
            continue
        f = dict(kv.split("=", 1) for kv in line.split()[1:])
        if f.get("call") == call and f.get("plan") == key and f.get("sha") == sha:
            return int(f["bytes"])
    return None


def plan_args(call):
    import rank_sum_residual_gb300 as farn
    p, xs, res, w, outs = call
    return (farn.FARN_F32 if p.partial_bytes == 4 else farn.FARN_BF16, p.W, p.T, p.H,
            [x.data_ptr() for x in xs], res.data_ptr(), w.data_ptr(),
            outs[0].data_ptr(), outs[1].data_ptr(),
            outs[2].data_ptr() if outs[2] is not None else 0,
            farn.FARN_PLAN_FP8_OUT if p.fp8_out else
            (farn.FARN_PLAN_NVFP4_OUT if p.nvfp4_out else 0))


def make_outputs(p, dev):
    """(reduced, residual_out, norm_out or None[, E4M3 bytes, row scales |
    E2M1 code bytes, E4M3 block scales])."""
    import torch
    outs = [torch.empty((p.T, p.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    outs.append(torch.empty((p.T, p.H), dtype=torch.bfloat16, device=dev)
                if p.norm_out else None)
    if p.fp8_out:
        outs.append(torch.empty((p.T, p.H), dtype=torch.uint8, device=dev))
        outs.append(torch.empty((p.T,), dtype=torch.float32, device=dev))
    if p.nvfp4_out:
        outs.append(torch.empty((p.T, p.H // 2), dtype=torch.uint8, device=dev))
        outs.append(torch.empty((p.T, p.H // 16), dtype=torch.uint8, device=dev))
    return tuple(outs)


def call_forward(p, xs, res, w, outs, ctx, stream):
    """One operator call through the binding of the C ABI."""
    import rank_sum_residual_gb300 as farn
    if p.kind == "moe_combine":
        ex, index, gates = xs
        farn.moe_combine(ex, index, gates, res, w, p.eps, out=outs, ctx=ctx, stream=stream)
        return
    if not p.fp8_out and not p.nvfp4_out:
        farn.forward(xs, res, w, p.eps, out=outs, ctx=ctx, stream=stream)
        return
    s = stream if stream is not None else __import__("torch").cuda.current_stream()
    if p.nvfp4_out:
        st = farn.farn_forward_nvfp4(
            (ctx or farn._context_for(res.device.index)).handle, [x.data_ptr() for x in xs],
            farn.FARN_F32 if p.partial_bytes == 4 else farn.FARN_BF16, len(xs), res.data_ptr(),
            w.data_ptr(), p.eps, p.T, p.H, p.tensor_scale, outs[0].data_ptr(),
            outs[1].data_ptr(), outs[2].data_ptr() if outs[2] is not None else 0,
            outs[3].data_ptr(), outs[4].data_ptr(), s.cuda_stream)
        if st != farn.FARN_OK:
            raise farn.FarnError(st, "farn_forward_nvfp4")
        return
    st = farn.farn_forward_quant(
        (ctx or farn._context_for(res.device.index)).handle, [x.data_ptr() for x in xs],
        farn.FARN_F32 if p.partial_bytes == 4 else farn.FARN_BF16, len(xs), res.data_ptr(),
        w.data_ptr(), p.eps, p.T, p.H, outs[0].data_ptr(), outs[1].data_ptr(),
        outs[2].data_ptr() if outs[2] is not None else 0, outs[3].data_ptr(),
        outs[4].data_ptr(), s.cuda_stream)
    if st != farn.FARN_OK:
        raise farn.FarnError(st, "farn_forward_quant")


def prepare_call(p, xs, res, w, outs, ctx, stream):
    """One call of the workload through the binding's prepared-call API:
    tensors checked and C-ABI arguments marshalled once, then each call is
    only the C call (the per-call host cost of a caller that keeps its
    buffers)."""
    import rank_sum_residual_gb300 as farn
    if p.kind == "moe_combine":
        ex, index, gates = xs
        return farn.prepare_moe_combine(ex, index, gates, res, w, p.eps, out=tuple(outs[:3]),
                                        ctx=ctx, stream=stream)
    if p.nvfp4_out:
        return farn.prepare_forward_nvfp4(xs, res, w, p.eps, p.tensor_scale, p.norm_out,
                                          out=tuple(outs), ctx=ctx, stream=stream)
    if p.fp8_out:
        return farn.prepare_forward_quant(xs, res, w, p.eps, p.norm_out, out=tuple(outs),
                                          ctx=ctx, stream=stream)
    return farn.prepare_forward(xs, res, w, p.eps, out=tuple(outs[:3]), ctx=ctx, stream=stream)


def time_calls_alone(problems, dev, ctx, l2_bytes, min_launches=64):
    """Mean launch duration of each call of a step, timed alone and from
    HBM: each call gets its own rotation of input/output copies, together
    at least twice the L2 size, laid out as one [copies, T, H] tensor per
    operand and launched back to back from one CUDA graph."""
    import torch
    import rank_sum_residual_gb300 as farn
    import synth
    out = []
    for p in problems:
        copies = max(2, math.ceil(2 * l2_bytes / p.algorithmic_bytes()))
        res = torch.empty((copies, p.T, p.H), dtype=torch.bfloat16, device=dev)
        w = torch.empty((p.H,), dtype=torch.bfloat16, device=dev)
        if p.kind == "moe_combine":
            ex = torch.empty((copies, p.T * p.W, p.H), dtype=torch.bfloat16, device=dev)
            synth.fill_device(ex, p.seed + 1, 0, p.x)
            index, gates = (torch.from_numpy(a).to(dev) for a in synth.moe_routing(p))
            ins = [(ex[c], index, gates) for c in range(copies)]
        else:
            xdt = torch.float32 if p.partial_bytes == 4 else torch.bfloat16
            xs = [torch.empty((copies, p.T, p.H), dtype=xdt, device=dev) for _ in range(p.W)]
            for r, x in enumerate(xs):
                synth.fill_device(x, p.seed + 1, r, p.x)
            ins = [[x[c] for x in xs] for c in range(copies)]
        synth.fill_device(res, p.seed + 1, synth.STREAM_RESIDUAL, p.residual)
        synth.fill_device(w, p.seed + 1, synth.STREAM_WEIGHT, p.weight)
        outs = [make_outputs(p, dev) for _ in range(copies)]
        reps = max(min_launches, copies)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                c = i % copies
                call_forward(p, ins[c], res[c], w, outs[c], ctx, None)
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            g.replay()
        e1.record()
        e1.synchronize()
        out.append(dict(call=p.name, T=p.T, W=p.W, H=p.H, bytes=p.algorithmic_bytes(),
                        count_per_step=1, launches_timed=3 * reps, rotating_copies=copies,
                        kernel_us=e0.elapsed_time(e1) / (3 * reps) * 1e3))
        del g, ins, res, w, outs
        torch.cuda.empty_cache()
    return out


def run_e2e(calls, problems, stream, dev, K, world, step_bytes):
    """Host buffers -> device -> farn_forward -> host, every step.

    A step's inputs sit in one pinned host buffer and its outputs land in
    one pinned host buffer, so each step is one host-to-device copy, the
    calls, and one device-to-host copy.  Two device buffer slots and three
    streams (copy in, compute, copy out) let step i+1's input copy and step
    i-1's output copy run while step i computes; every step's copies are
    inside the timed region."""
    import torch
    import rank_sum_residual_gb300 as farn

    # inputs and outputs packed as bytes (fp32 partials, E4M3 outputs)
    in_bytes = sum(p.read_bytes() for p in problems)
    out_bytes = sum(p.write_bytes() for p in problems)
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    host_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    off = 0
    for p, xs, res, w, outs in calls:          # the step's inputs, packed
        for t in (*xs, res, w):                # (expert_out, index, gates) for MoE
            b = t.reshape(-1).view(torch.uint8)
            host_in[off:off + b.numel()].copy_(b)
            off += b.numel()
    slots = []
    for _ in range(2):
        dev_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        dev_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        views, cur = [], {"in": 0, "out": 0}

        def take(buf, key, nbytes, dtype, shape):
            t = buf[cur[key]:cur[key] + nbytes].view(dtype).view(*shape)
            cur[key] += nbytes
            return t
        for p in problems:
            n = p.T * p.H
            if p.kind == "moe_combine":
                xs = (take(dev_in, "in", n * p.W * 2, torch.bfloat16, (p.T * p.W, p.H)),
                      take(dev_in, "in", p.T * p.W * 4, torch.int32, (p.T, p.W)),
                      take(dev_in, "in", p.T * p.W * 4, torch.float32, (p.T, p.W)))
            else:
                xdt = torch.float32 if p.partial_bytes == 4 else torch.bfloat16
                xs = [take(dev_in, "in", n * p.partial_bytes, xdt, (p.T, p.H))
                      for _ in range(p.W)]
            res = take(dev_in, "in", n * 2, torch.bfloat16, (p.T, p.H))
            w = take(dev_in, "in", p.H * 2, torch.bfloat16, (p.H,))
            outs = [take(dev_out, "out", n * 2, torch.bfloat16, (p.T, p.H)) for _ in range(2)]
            outs.append(take(dev_out, "out", n * 2, torch.bfloat16, (p.T, p.H))
                        if p.norm_out else None)
            if p.fp8_out:
                outs.append(take(dev_out, "out", n, torch.uint8, (p.T, p.H)))
                outs.append(take(dev_out, "out", 4 * p.T, torch.float32, (p.T,)))
            if p.nvfp4_out:
                outs.append(take(dev_out, "out", n // 2, torch.uint8, (p.T, p.H // 2)))
                outs.append(take(dev_out, "out", n // 16, torch.uint8, (p.T, p.H // 16)))
            views.append((p, xs, res, w, tuple(outs)))
        slots.append((dev_in, dev_out, views))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_comp = stream
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    for k in ev:
        for e in ev[k]:
            e.record(s_comp)

    # each slot's calls, marshalled once: per step only the C-ABI calls run
    prepared = [[prepare_call(p, xs, res, w, outs, None, s_comp)
                 for p, xs, res, w, outs in slots[j][2]] for j in range(2)]

    def e2e_step(i):
        j = i % 2
        dev_in, dev_out, views = slots[j]
        s_in.wait_event(ev["comp"][j])             # slot's inputs no longer read
        with torch.cuda.stream(s_in):
            dev_in.copy_(host_in, non_blocking=True)
        ev["in"][j].record(s_in)
        s_comp.wait_event(ev["in"][j])
        s_comp.wait_event(ev["out"][j])            # slot's outputs copied out
        for call in prepared[j]:
            call()
        ev["comp"][j].record(s_comp)
        s_out.wait_event(ev["comp"][j])
        with torch.cuda.stream(s_out):
            host_out[j].copy_(dev_out, non_blocking=True)
        ev["out"][j].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(6):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    per = (time.perf_counter() - t0) / 6
    Ke = int(min(K, max(10, 1.0 / max(per, 1e-7))))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(Ke):
        e2e_step(i)
    s_in.wait_event(ev["out"][(Ke - 1) % 2])
    s_in.wait_event(ev["out"][Ke % 2])
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    # the last step's outputs really came back
    assert torch.equal(host_out[(Ke - 1) % 2][-8:], slots[(Ke - 1) % 2][1][-8:].cpu())
    return {"value": world * step_bytes * Ke / (ms / 1e3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
            "steps": Ke, "ms_per_step": ms / Ke,
            "path": "per step: one pinned-host -> device copy of all inputs, "
                    "every call through the binding's prepared calls (C ABI, arguments "
                    "checked and marshalled once), one "
                    "device -> pinned-host copy of all three outputs; copy-in, compute "
                    "and copy-out on three streams over two buffer slots"}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
