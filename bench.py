#!/usr/bin/env python3
"""Benchmark of the fused ZeRO reduce-scatter + Adam + all-gather step.

One step = one call of ``zero_adam_step`` (all P simulated ranks' shards:
reduce-scatter of the fp16 gradients, fp32 Adam, fp16 cast, write into the
gathered parameter vector) over one batch of synthetic gradients.  The
default workload is the largest that fits one GPU: N = 1.3e9 parameters laid
out as 24 transformer blocks at d = 2048 plus an embedding, P = 16 ranks,
ZeRO-2, standard Adam, gradients ~ N(0, 1e-4).

Printed: one JSON line (rank 0).  ``value`` is parameters updated per second
over the whole job with every input resident in HBM; ``e2e`` is the same
metric with each step's gradients copied from pinned host memory and the
gathered fp16 parameters copied back inside the timed region;
``roofline`` rates the fused kernel against the measured HBM copy bandwidth;
``per_config`` times every other workload (the 1,000,003-element vector, the
GPT-2-small vector, one shard of a 7.5e9 model at P = 64 and both folded Adam
readings at P = 32) in the same run, each with its own roofline fraction;
``cpu_baseline`` times the CPU oracle on the host cores, single-threaded and
on every core the process may use, on bounded samples of every workload.

``--impl reference`` times the CPU oracle instead (the only other
implementation of this step), on the same workload and metric.

Multi-GPU (torchrun): every rank runs its own independent replica of the
whole simulated step on its own GPU -- the path has no exchange between
GPUs -- and ``value`` counts all ranks' parameters over the slowest rank's
time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024   # GB300's L2 (nominal)
DEFAULT_STEPS = {"tiny": 20000, "gpt2s": 2500, "tf1p3b": 200, "shard7p5b": 800, "folded": 600}
# every workload with each Adam reading it runs; the headline is one of them,
# the rest go to the line's per_config block
ALL_CONFIGS = (("tiny", 0), ("gpt2s", 0), ("tf1p3b", 0), ("shard7p5b", 0), ("folded", 1), ("folded", 2))
# also timed in per_config: the 7.5B shard in its natural packed layout, rank
# stride M = 117,187,500 elements (4 mod 8: the vector kernel at width 4)
UNPADDED_CONFIGS = (("shard7p5b", 0),)
# timed steps of a per_config leg: at least this many (about 0.2 s of GPU time)
PER_CONFIG_MIN_STEPS = {"tiny": 2000, "gpt2s": 250, "tf1p3b": 20, "shard7p5b": 80, "folded": 60}
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SRC = os.path.join(ROOT, "zero_sharded_mixed_shard_gb300", "csrc", "step.cu")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="tf1p3b",
                    choices=("tiny", "gpt2s", "tf1p3b", "shard7p5b", "folded"))
    ap.add_argument("--mode", type=int, default=None, help="Adam reading (default: the workload's first)")
    ap.add_argument("--ranks", type=int, default=None,
                    help="override the workload's rank count P (whole-vector workloads; N unchanged)")
    ap.add_argument("--elements", type=int, default=None,
                    help="override the workload's element count N (whole-vector workloads; a smaller case "
                         "of the same kernel, e.g. for a profiler capture)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time the chosen workload only (no per_config block)")
    ap.add_argument("--unpadded-stride", action="store_true",
                    help="rank stride = the elements of a rank's slice, not rounded up to a multiple of 8 "
                         "(rows off the 16-byte phase: the phased pipeline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=24.0,
                    help="wall time budget of the CPU-oracle leg (all of its runs together)")
    ap.add_argument("--overlap", action="store_true",
                    help="time the bucketed step overlapped with a synthetic backward instead")
    ap.add_argument("--bucket-elems", type=int, default=1 << 24)
    ap.add_argument("--backward-k", type=int, default=2048,
                    help="inner dimension of the synthetic backward's GEMMs")
    ap.add_argument("--step-priority", choices=("high", "normal"), default="high",
                    help="priority of the step's stream in the overlap leg")
    ap.add_argument("--step-sms", type=int, default=0,
                    help="overlap leg: SMs the step of every bucket but the last may occupy "
                         "(0 = all); the last bucket, which nothing hides, runs uncapped")
    ap.add_argument("--gemm-carveout", type=int, default=0,
                    help="overlap leg: SMs the backward's cuBLAS GEMMs leave free")
    ap.add_argument("--offload", action="store_true",
                    help="time the ZeRO-Offload step (update on the host CPU) instead")
    ap.add_argument("--mlp4", action="store_true",
                    help="time the layer-pipelined ZeRO-3 step of the 4-layer scalar MLP instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload]
    return args


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU under torchrun)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def all_true(self, ok: bool, device=None) -> bool:
        """True on every rank iff ``ok`` is true on every rank."""
        if not self.pg:
            return ok
        import torch
        t = torch.tensor([1 if ok else 0], dtype=torch.int32, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MIN)
        return bool(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.out = None
        self.gpu = gpu_index
        self.period = period_ms

    def start(self):
        import tempfile
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, *windows) -> list:
        """Stop sampling; for each (t0, t1) host-time window, the clocks seen in it."""
        if self.proc is None:
            return [{"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                     "note": "nvidia-smi unavailable"} for _ in windows]
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        text = self.out.read()
        self.out.close()
        os.unlink(self.out.name)
        return [parse_clock_csv(text, t0, t1) for t0, t1 in windows]


def parse_clock_csv(text: str, t0: float, t1: float) -> dict:
    """Median SM clock, max clock and active slowdown reasons of the samples
    taken between host times t0 and t1 (nvidia-smi's local timestamps)."""
    rows = []
    for line in text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            stamp = parts[0]
            ts = time.mktime(time.strptime(stamp.split(".")[0], "%Y/%m/%d %H:%M:%S"))
            if "." in stamp:
                ts += float("0." + stamp.split(".")[1])
            rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
        except (ValueError, IndexError):
            continue
    inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    reasons = sorted({names[i] for r in inside for i, s in enumerate(r[3]) if s == "Active"})
    return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
            "sm_max_mhz": max((r[2] for r in inside), default=None),
            "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------

def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the kernel source's code: comments and blank space taken out,
    so a summary stays valid across edits that change no code."""
    import re
    with open(KERNEL_SRC, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)      # block comments
    text = re.sub(r"//[^\n]*", " ", text)                    # line comments
    text = " ".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "zero_fused_step_tma_kernel", mode: int | None = None
                     ) -> float | None:
    """DRAM bytes per launch from the committed ncu summary of this workload
    (the Adam reading's own figure where the summary has one per mode), if
    it was taken on the current kernel source and of the kernel the step
    launches now."""
    path = os.path.join(PROFILE_DIR, f"zero_fused_step_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != kernel_source_hash():
            return None
        if not kv.get("kernel", "").startswith(kernel.split(" ")[0]):
            return None
        if mode is not None and f"traffic_bytes_per_launch_mode{mode}" in kv:
            return float(kv[f"traffic_bytes_per_launch_mode{mode}"])
        return float(kv["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# the CPU oracle leg (used by cpu_baseline and by --impl reference)
# ---------------------------------------------------------------------------

def host_cores() -> tuple[int, int]:
    """(logical CPUs of the machine -- what std::thread::hardware_concurrency
    reports --, CPUs this process may run on, from its affinity mask)."""
    hw = os.cpu_count() or 1
    try:
        allowed = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        allowed = hw
    return hw, allowed


def oracle_inputs(wl, sample: int, draw: int | None = None):
    """Seeded host inputs for ``sample`` elements of the workload, all P
    ranks.  With ``draw`` < sample, a draw of that many elements is repeated
    to fill the sample (the oracle's time does not depend on the values
    beyond their mix, which the repeated draw keeps)."""
    import numpy as np

    from zero_sharded_mixed_shard_gb300 import synth
    n = sample if draw is None else min(draw, sample)
    codes = synth.np_grads(wl.P, n, n, wl.grad_sigma, wl.seed, wl.heavy_tail_frac, wl.zero_frac)
    w, m, v, _ = synth.np_state(n, wl.seed, wl.master_sigma)
    if n < sample:
        reps = -(-sample // n)
        codes = np.ascontiguousarray(np.tile(codes.reshape(wl.P, n), (1, reps))[:, :sample]).reshape(-1)
        w = np.ascontiguousarray(np.tile(w, reps)[:sample])
        m = np.zeros(sample, np.float32)
        v = np.zeros(sample, np.float32)
    return codes, w, m, v


def oracle_rate(wl, mode: int, budget_s: float, sample: int | None = None, steps: int | None = None,
                threads: int | None = None, draw: int | None = None):
    """Time the oracle (as it stands) on the first ``sample`` elements of
    the workload, all P ranks, ``threads`` host threads (default: every CPU
    the process may use), consecutive steps until ``budget_s`` has passed
    (at least one) or ``steps`` steps.  Returns (params/s, threads, sample,
    per-step seconds list)."""
    import numpy as np

    import oracle
    oracle.build()
    if threads is None:
        threads = host_cores()[1]
    if sample is None:
        sample = min(wl.elems, 1 << 24)
    codes, w, m, v = oracle_inputs(wl, sample, draw)
    out = np.empty(sample, np.uint16)
    times = []
    t = 0
    start = time.perf_counter()
    while True:
        t += 1
        t0 = time.perf_counter()
        oracle.adam_elems(codes, sample, wl.P, w, m, v, t, wl.lr, wl.b1, wl.b2, wl.eps, mode,
                          threads=threads, params_out=out)
        times.append(time.perf_counter() - t0)
        if steps is not None:
            if t >= steps:
                break
        elif time.perf_counter() - start >= budget_s:
            break
    return sample * len(times) / sum(times), threads, sample, times


def cpu_baseline_leg(wl, mode: int, budget_s: float, configs=()) -> dict:
    """The oracle on the host cores: the headline workload on every allowed
    CPU and on one thread, and a per-element rate for each other workload.
    The tiny and GPT-2-small workloads are timed on whole steps; the larger
    ones on their first 2^22 elements, extrapolated to a whole step and
    labelled so (elements never interact, so the per-element cost is the
    same everywhere in the vector)."""
    from zero_sharded_mixed_shard_gb300 import synth
    hw, allowed = host_cores()
    rate, threads, sample, times = oracle_rate(wl, mode, 0.35 * budget_s)
    one_sample = min(wl.elems, 1 << 22)
    rate1, _, _, times1 = oracle_rate(wl, mode, 0.2 * budget_s, sample=one_sample, threads=1)
    out = {"value": rate, "unit": "params/s", "cores": threads, "kind": "oracle",
           "sample": f"elements [0, {sample}) of the {wl.name} workload, all {wl.P} ranks, "
                     f"{len(times)} consecutive steps in {sum(times):.1f} s on {threads} threads",
           "hardware_concurrency": hw, "affinity_cores": allowed, "threads_used": threads,
           "single_thread": {"value": rate1, "unit": "params/s", "threads_used": 1,
                             "sample": f"elements [0, {one_sample}) of the {wl.name} workload, "
                                       f"{len(times1)} steps in {sum(times1):.1f} s"},
           "full_step_s_extrapolated": wl.elems / rate}
    per = {}
    share = 0.45 * budget_s / max(1, len(configs))
    for cwl, cmode in configs:
        whole = cwl.elems * cwl.P <= (1 << 30)    # tiny and gpt2s: whole steps
        n = cwl.elems if whole else min(cwl.elems, 1 << 22)
        r, th, n, ts = oracle_rate(cwl, cmode, share, sample=n, draw=min(n, 1 << 22))
        per[f"{cwl.name}/mode{cmode}"] = {
            "value": r, "unit": "params/s", "threads_used": th,
            "gbs": r * synth.bytes_per_elem(cwl.P, cmode) / 1e9,
            "kind": "whole step" if whole else "elements [0, 2^22), extrapolated to a whole step",
            "sample": (f"all {n} elements" if whole else f"elements [0, {n})")
                      + f", {len(ts)} steps in {sum(ts):.1f} s"
                      + (" (a 2^22-element draw repeated to fill the vector)" if whole and n > (1 << 22) else ""),
            "step_s": cwl.elems / r}
    if per:
        out["per_config"] = per
    return out


def run_reference(args, wl, mode, dist):
    """--impl reference: the CPU oracle on the same workload, rank 0 only."""
    from zero_sharded_mixed_shard_gb300 import synth
    if dist.rank != 0:
        return 0
    # size each step's sample so the whole run stays within ~90 s of host time
    rate, cores, _, _ = oracle_rate(wl, mode, 0.0, sample=min(wl.elems, 1 << 22), steps=1)
    per_step = 90.0 / (args.steps + args.warmup)
    sample = int(min(wl.elems, 1 << 24, max(4096, rate * per_step)))
    _, cores, sample, times = oracle_rate(wl, mode, 0.0, sample=sample,
                                          steps=args.steps + args.warmup)
    timed = times[args.warmup:]
    sec = sum(timed)
    value = sample * len(timed) / sec
    hw, allowed = host_cores()
    note = (f"each step runs the oracle on elements [0, {sample}) of the {wl.name} workload, all "
            f"{wl.P} ranks; params/s counts those elements")
    line = {
        "impl": "reference",
        "metric": "params updated/sec and achieved HBM GB/s (% of GB300 peak) per Adam step",
        "value": value, "unit": "params/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(timed), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(wl, mode, l2_flush_bytes=l2_flush_for(wl, mode)),
        "sample": note,
        "achieved_gbs": value * synth.bytes_per_elem(wl.P, mode) / 1e9,
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": cores, "kind": "oracle",
                         "sample": note, "hardware_concurrency": hw, "affinity_cores": allowed,
                         "threads_used": cores},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_flush_for(wl, mode) -> int | None:
    """Bytes written between timed steps to flush L2, or None: a step that
    moves less than twice the L2 would partly run from L2 when repeated, so
    a buffer of 4x the L2 is written between its timed steps, then another
    one of 4x the L2 is read (so the L2 holds clean lines of neither the
    step's buffers nor the flush's: the step pays for no write-back of the
    flush's dirty lines), and only the steps themselves are timed."""
    from zero_sharded_mixed_shard_gb300 import synth
    alg = wl.elems * synth.bytes_per_elem(wl.P, mode)
    return 4 * L2_BYTES if alg < 2 * L2_BYTES else None


def workload_config(wl, mode, l2_flush_bytes=None):
    from zero_sharded_mixed_shard_gb300 import synth
    step_gb = wl.elems * synth.bytes_per_elem(wl.P, mode) / 1e9
    if l2_flush_bytes:
        l2 = (f"L2 flushed between timed steps ({l2_flush_bytes / 1e6:.0f} MB written, then "
              f"{l2_flush_bytes / 1e6:.0f} MB read; a step moves only {step_gb * 1e3:.1f} MB); "
              f"value from the summed per-step event times")
    else:
        l2 = f"inputs larger than L2: {step_gb:.2f} GB moved per step"
    cfg = {"workload": f"{wl.name}: N={wl.N:,} P={wl.P} ZeRO-{wl.stage} "
                       f"{'shard ' + str(wl.shard) + ' only, ' if wl.shard is not None else ''}"
                       f"Adam mode {mode}",
           "N": wl.N, "elements_per_step": wl.elems, "P": wl.P, "stage": wl.stage, "mode": mode,
           "rank_stride": wl.rank_stride(True), "bytes_per_elem": synth.bytes_per_elem(wl.P, mode),
           "l2": l2}
    return cfg


def kernel_label(plan) -> str:
    return ("zero_fused_step_tma_kernel" if plan["kernel"] == "bulk"
            else f"zero_fused_step_kernel (vector width {plan['vector_width']})")


class Timed:
    """One workload on the device: its buffers, a step function and the
    timing of K steps after W warm-up steps (CUDA events on the launching
    stream, one pair per step)."""

    def __init__(self, z, wl, mode, dist, device, stream, padded=True, flush=True):
        import torch

        from zero_sharded_mixed_shard_gb300 import synth
        self.z, self.wl, self.mode, self.dist, self.stream = z, wl, mode, dist, stream
        E, P = wl.elems, wl.P
        self.stride = wl.rank_stride(padded)
        self.g = synth.torch_grads(P, E, self.stride, wl.grad_sigma, wl.seed + 17 * dist.rank, device,
                                   wl.heavy_tail_frac, wl.zero_frac, step=1)
        self.master, self.m, self.v, self.params = synth.torch_state(E, wl.seed + 17 * dist.rank, device,
                                                                     wl.master_sigma)
        # the kernel the step launches (the shard call is a step of E elements
        # from the same buffers, so it takes the same decision)
        self.plan = z.zero_step_plan(self.g, self.stride, self.master, self.m, self.v, self.params, E, P,
                                     wl.stage, mode)
        self.alg_bytes = E * synth.bytes_per_elem(P, mode)
        fb = l2_flush_for(wl, mode) if flush else None
        self.flush = torch.empty(fb, dtype=torch.uint8, device=device) if fb else None
        self.flush_read = torch.ones(fb // 4, dtype=torch.float32, device=device) if fb else None
        self.t = 0

    def flush_l2(self):
        if self.flush is not None:
            self.flush.zero_()
            self.flush_read.sum()

    def step(self, g=None):
        wl, z = self.wl, self.z
        self.t += 1
        g = self.g if g is None else g
        if wl.shard is None:
            z.zero_adam_step(g, self.stride, self.master, self.m, self.v, self.params, wl.N, wl.P,
                             wl.stage, self.t, wl.lr, wl.b1, wl.b2, wl.eps, self.mode, self.stream)
        else:
            z.zero_adam_step_shard(g, self.stride, 0, wl.shard, self.master, self.m, self.v,
                                   self.params, wl.N, wl.P, wl.stage, self.t, wl.lr, wl.b1, wl.b2,
                                   wl.eps, self.mode, self.stream)

    def warm(self, W):
        import torch
        for _ in range(W):
            self.flush_l2()
            self.step()
        torch.cuda.synchronize()

    def run(self, K):
        """Time K steps (the caller brackets them with barrier + synchronize).
        Returns (region ms, mean launch ms); with an L2 flush between steps
        the region is the sum of the steps' own times."""
        import torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            self.flush_l2()
            starts[i].record(self.stream)
            self.step()
            ends[i].record(self.stream)
        torch.cuda.synchronize()
        launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        region_ms = starts[0].elapsed_time(ends[-1]) if self.flush is None else sum(launch_ms)
        return region_ms, sum(launch_ms) / K

    def free(self):
        import torch
        self.g = self.master = self.m = self.v = self.params = self.flush = self.flush_read = None
        torch.cuda.empty_cache()


def one_element_step_ms(z, wl, mode, K, dist, device, stream) -> float:
    """Mean event-to-event time of a step of ONE element with the workload's
    P and mode, under the same L2 flush: the fixed cost of a launch through
    the library (enqueue to completion), against which a small workload's
    own time can be read."""
    one = dataclasses.replace(wl, N=1, shard=None, tensors=None, name=wl.name + "-N1")
    leg = Timed(z, one, mode, dist, device, stream)   # flushed like any step below 2x the L2
    leg.warm(3)
    _, ms = leg.run(K)
    leg.free()
    return ms


def ring_step_ms(z, wl, mode, K, dist, device, stream) -> tuple[float, int]:
    """Steps of R independent copies of a small workload, round-robin and
    back to back (one event pair around all K steps, no flush): R is chosen
    so the copies together are 4x the L2, so every step's inputs have left
    L2 by the time its copy comes round again.  Returns (ms per step, R)."""
    import torch
    from zero_sharded_mixed_shard_gb300 import synth
    R = max(2, -(-4 * L2_BYTES // (wl.elems * synth.bytes_per_elem(wl.P, mode))))
    legs = [Timed(z, wl, mode, dist, device, stream, flush=False) for _ in range(R)]
    for leg in legs:
        leg.step()
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        legs[i % R].step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(e0.elapsed_time(e1) / K, device)
    for leg in legs:
        leg.free()
    return ms, R


def roofline_entry(wl, mode, plan, alg_bytes, mean_launch_ms):
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (mean_launch_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": profiled_traffic(wl.name, kernel_label(plan), mode),
            "kernel": kernel_label(plan), "ctas": plan["ctas"],
            "peak_kind": f"{peak_kind} HBM copy bandwidth",
            "algorithmic_bytes_per_launch": alg_bytes, "mean_launch_ms": mean_launch_ms}


def run_ours(args, wl, mode, dist):
    import torch

    import zero_sharded_mixed_shard_gb300 as z
    from zero_sharded_mixed_shard_gb300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the fused step has no CPU path)")
    torch.cuda.set_device(dist.local_rank)
    dist.init("nccl")
    device = torch.device("cuda", dist.local_rank)
    z.lib()
    stream = torch.cuda.current_stream(device)

    head = Timed(z, wl, mode, dist, device, stream, padded=not args.unpadded_stride)
    head.warm(args.warmup)
    K = args.steps
    sampler = ClockSampler(dist.local_rank)
    if dist.rank == 0:
        sampler.start()
    dist.barrier()
    torch.cuda.synchronize()
    h0 = time.time()
    region_ms, mean_launch_ms = head.run(K)
    h1 = time.time()
    dist.barrier()
    region_ms = dist.max(region_ms, device)
    mean_launch_ms = dist.max(mean_launch_ms, device)
    E = wl.elems
    value = E * K * dist.world / (region_ms / 1e3)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(head, device, dist)
    flush_bytes = None if head.flush is None else head.flush.numel()
    plan, alg_bytes = head.plan, head.alg_bytes
    head.free()
    del head

    # every other workload, in the same run and under the same clock sampler
    per_config = None
    p0 = p1 = None
    if not args.no_per_config and args.ranks is None and args.elements is None and not args.unpadded_stride:
        per_config = {}
        p0 = time.time()
        legs = [(n, cm, True) for n, cm in ALL_CONFIGS if (n, cm) != (wl.name, mode)]
        legs += [(n, cm, False) for n, cm in UNPADDED_CONFIGS]
        for name, cmode, padded in legs:
            cwl = synth.WORKLOADS[name]
            if not padded:
                cwl = dataclasses.replace(cwl, name=f"{name}-unpadded")
            leg = Timed(z, cwl, cmode, dist, device, stream, padded=padded)
            leg.warm(args.warmup)
            ck = max(K, PER_CONFIG_MIN_STEPS[name])
            dist.barrier()
            torch.cuda.synchronize()
            r_ms, l_ms = leg.run(ck)
            dist.barrier()
            r_ms, l_ms = dist.max(r_ms, device), dist.max(l_ms, device)
            extra = {}
            if leg.flush is not None:   # a small workload: how much of its time is the launch
                floor = dist.max(one_element_step_ms(z, cwl, cmode, ck, dist, device, stream), device)
                ring_ms, ring_r = ring_step_ms(z, cwl, cmode, ck, dist, device, stream)
                extra = {"one_element_step_ms": floor,
                         "gbs_above_one_element_step": leg.alg_bytes / ((l_ms - floor) / 1e3) / 1e9
                         if l_ms > floor else None,
                         "back_to_back": {"ms_per_step": ring_ms, "copies": ring_r,
                                          "gbs": leg.alg_bytes / (ring_ms / 1e3) / 1e9,
                                          "how": f"{ck} steps round-robin over {ring_r} independent copies "
                                                 "of the workload (4x the L2 together), one event pair "
                                                 "around them all, no flush"}}
            per_config[f"{name}/mode{cmode}" + ("" if padded else "/unpadded")] = {
                "workload": workload_config(cwl, cmode, None if leg.flush is None else leg.flush.numel())["workload"]
                            + ("" if padded else f", rank stride {leg.stride:,}"),
                "value": cwl.elems * ck * dist.world / (r_ms / 1e3), "unit": "params/s", "steps": ck,
                "ms_per_step": r_ms / ck,
                "roofline": roofline_entry(cwl, cmode, leg.plan, leg.alg_bytes, l_ms),
                "l2": "flushed between timed steps" if leg.flush is not None else "inputs larger than L2",
                **extra}
            leg.free()
            del leg
        p1 = time.time()
    clocks_list = sampler.stop((h0, h1), *([(p0, p1)] if p0 is not None else [])) if dist.rank == 0 else None
    if per_config is not None and clocks_list:
        per_config["clocks"] = clocks_list[1] if len(clocks_list) > 1 else None

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        others = [] if per_config is None else [
            (synth.WORKLOADS[n], cm) for n, cm in ALL_CONFIGS if (n, cm) != (wl.name, mode)]
        cpu = cpu_baseline_leg(wl, mode, args.cpu_seconds, others)

    if dist.rank == 0:
        line = {
            "metric": "params updated/sec and achieved HBM GB/s (% of GB300 peak) per Adam step",
            "value": value, "unit": "params/s", "n_gpus": dist.world, "steps": K,
            "warmup": args.warmup, "ms_per_step": region_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "io_dtypes": "fp16 gradients and parameters, fp32 master/m/v",
            "data": "synthetic (seeded device RNG)",
            "config": dict(workload_config(wl, mode, l2_flush_bytes=flush_bytes),
                           **({"rank_stride": wl.rank_stride(False)} if args.unpadded_stride else {})),
            "achieved_hbm_gbs": alg_bytes * K * dist.world / (region_ms / 1e3) / 1e9,
            "pct_of_nominal_8tbs": 100 * alg_bytes * K / (region_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
            "roofline": roofline_entry(wl, mode, plan, alg_bytes, mean_launch_ms),
            "gpu_launches": K,
            "clocks": clocks_list[0] if clocks_list else None,
            "e2e": e2e,
            "per_config": per_config,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def run_e2e(head, device, dist):
    """Each step: pinned host gradients -> device, the step, gathered fp16
    parameters -> pinned host; all inside the timed region.

    Steps are pipelined the way a training loop would: the upload of step
    k+1's gradients (into the second of two device buffers, on its own
    stream) runs while step k's kernel and the download of its parameters
    run; step k+1's kernel waits for its upload and for the download of
    step k's parameters (which it overwrites).  The number of steps is
    bounded so the leg takes about 5 s (the upload is limited by the host
    link, ~200 GB/s)."""
    import torch
    g, params, stream = head.g, head.params, head.stream
    host_g = host_p = None
    why = ""
    try:
        host_g = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
        host_p = torch.empty(params.shape, dtype=params.dtype, pin_memory=True)
    except RuntimeError as exc:   # the host could not page-lock that much memory
        why = f"pinned host buffers: {exc}"[:200]
    # every rank runs the leg or none does (its barriers must pair up)
    if not dist.all_true(host_p is not None, device):
        del host_g, host_p
        return {"value": None, "unit": "params/s",
                "unavailable": why or "another rank could not page-lock its host buffers"}
    host_g.copy_(g)
    h2d = host_g.numel() * host_g.element_size()
    K_e2e = max(3, min(100, int(5.0 / (h2d / 200e9 + 1e-4))))
    dev_g = [g, torch.empty_like(g)]
    up = torch.cuda.Stream(device)
    down = torch.cuda.Stream(device)
    for _ in range(2):   # warm the copy engines
        dev_g[1].copy_(host_g, non_blocking=True)
        host_p.copy_(params, non_blocking=True)
    torch.cuda.synchronize()
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    downloaded = torch.cuda.Event()
    for k in range(2):
        consumed[k].record(stream)
    downloaded.record(down)
    # upload of step 0
    with torch.cuda.stream(up):
        dev_g[0].copy_(host_g, non_blocking=True)
        uploaded[0].record(up)
    for k in range(K_e2e):
        b = k % 2
        if k + 1 < K_e2e:        # the next step's upload, into the other buffer
            nb = (k + 1) % 2
            up.wait_event(consumed[nb])
            with torch.cuda.stream(up):
                dev_g[nb].copy_(host_g, non_blocking=True)
                uploaded[nb].record(up)
        stream.wait_event(uploaded[b])
        stream.wait_event(downloaded)        # the previous parameters have left
        head.step(dev_g[b])
        consumed[b].record(stream)
        down.wait_event(consumed[b])
        with torch.cuda.stream(down):
            host_p.copy_(params, non_blocking=True)
            downloaded.record(down)
    stream.wait_event(downloaded)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(e0.elapsed_time(e1), device)
    out = {"value": head.wl.elems * K_e2e * dist.world / (ms / 1e3), "unit": "params/s",
           "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": host_p.numel() * host_p.element_size(),
           "steps": K_e2e, "ms_per_step": ms / K_e2e,
           "pipelining": "upload of step k+1 overlaps step k's kernel and download"}
    del dev_g, host_g, host_p
    return out


def run_overlap(args, wl, mode, dist):
    """Bucketed step on a second stream behind a synthetic backward.

    The backward pass is stood in for by one GEMM per bucket per rank,
    dW = X_r @ Y (X_r: [L/768, k], Y: [k, 768], fp16 on the tensor cores),
    written straight into rank r's gradient slice of the bucket, buckets in
    backward order.  Reported: the backward alone, the whole step alone, the
    two back to back on one stream, and the bucketed step on its own stream
    waiting on one event per bucket; ``value`` is the fraction of the step's
    time hidden behind the backward."""
    import torch

    import zero_sharded_mixed_shard_gb300 as z
    from zero_sharded_mixed_shard_gb300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the fused step has no CPU path)")
    if wl.tensors is None or wl.shard is not None or any(n % 768 for n in wl.tensors):
        raise SystemExit("--overlap needs a whole-vector workload with 768-multiple tensors (gpt2s)")
    torch.cuda.set_device(dist.local_rank)
    dist.init("nccl")
    dev = torch.device("cuda", dist.local_rank)
    P, N = wl.P, wl.N
    stride = wl.rank_stride(True)
    buckets = z.zero_plan_buckets(list(wl.tensors), args.bucket_elems, backward_order=True)
    g = torch.zeros((P, stride), dtype=torch.float16, device=dev)
    state = synth.torch_state(N, wl.seed, dev, wl.master_sigma)
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed)
    k = args.backward_k
    rows_max = max((e - b) // 768 for b, e, _, _ in buckets)
    X = [torch.randn(rows_max, k, generator=gen, device=dev).half() for _ in range(P)]
    Y = (torch.randn(k, 768, generator=gen, device=dev) * (1e-3 / k ** 0.5)).half()
    prod_stream = torch.cuda.Stream(dev)
    # a higher-priority stream lets the step's CTAs take SMs as the backward's
    # CTAs retire instead of queueing behind every later GEMM
    step_stream = torch.cuda.Stream(dev, priority=-1 if args.step_priority == "high" else 0)
    t_counter = [0]

    carve = args.gemm_carveout
    if carve and not hasattr(torch._C, "_set_sm_carveout_experimental"):
        raise SystemExit("--gemm-carveout needs torch._C._set_sm_carveout_experimental")

    def set_carveout(n):
        if carve:
            torch._C._set_sm_carveout_experimental(n if n else None)

    def backward(stream, events=None):
        with torch.cuda.stream(stream):
            for i, (b, e, _, _) in enumerate(buckets):
                rows = (e - b) // 768
                for r in range(P):
                    torch.mm(X[r][:rows], Y, out=g[r, b:e].view(rows, 768))
                if events is not None:
                    events[i].record(stream)

    def step_whole(stream):
        t_counter[0] += 1
        z.zero_adam_step(g, stride, *state, N, P, wl.stage, t_counter[0], wl.lr, wl.b1, wl.b2,
                         wl.eps, mode, stream)

    def step_bucketed(stream, events):
        t_counter[0] += 1
        args_ = (g, stride, *state, N, P, wl.stage, t_counter[0], wl.lr, wl.b1, wl.b2, wl.eps, mode)
        if args.step_sms and len(buckets) > 1:
            prev = z.zero_set_step_max_sms(args.step_sms)
            try:
                z.zero_adam_step_bucketed(*args_, buckets[:-1], ready_events=events[:-1],
                                          stream=stream)
            finally:
                z.zero_set_step_max_sms(prev)
            z.zero_adam_step_bucketed(*args_, buckets[-1:], ready_events=events[-1:],
                                      stream=stream)
        else:
            z.zero_adam_step_bucketed(*args_, buckets, ready_events=events, stream=stream)

    def timed(fn, reps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(step_stream)
        for _ in range(reps):
            fn()
        done = torch.cuda.Event()
        done.record(prod_stream)
        step_stream.wait_event(done)
        e1.record(step_stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def join(a, b):
        ev = torch.cuda.Event()
        ev.record(a)
        b.wait_event(ev)

    reps = max(3, min(args.steps, 50))

    def only_backward():
        join(step_stream, prod_stream)
        backward(prod_stream)

    def only_backward_carved():
        join(step_stream, prod_stream)
        set_carveout(carve)
        backward(prod_stream)
        set_carveout(0)

    def only_step():
        join(prod_stream, step_stream)
        step_whole(step_stream)

    def serial():
        join(step_stream, prod_stream)
        backward(prod_stream)
        step_whole(prod_stream)

    def overlapped():
        join(step_stream, prod_stream)
        events = [torch.cuda.Event() for _ in buckets]
        set_carveout(carve)
        backward(prod_stream, events)
        set_carveout(0)
        step_bucketed(step_stream, events)

    t_b = timed(only_backward, reps)
    t_s = timed(only_step, reps)
    t_serial = timed(serial, reps)
    t_over = timed(overlapped, reps)
    t_b_carved = timed(only_backward_carved, reps) if carve else t_b
    hidden = (t_serial - t_over) / t_s
    if dist.rank == 0:
        line = {
            "metric": "fraction of the optimizer step hidden behind a synthetic backward",
            "value": hidden, "unit": "fraction", "n_gpus": dist.world, "steps": reps,
            "warmup": args.warmup, "higher_is_better": True, "dtype": "f32",
            "data": "synthetic", "config": dict(workload_config(wl, mode),
                                                buckets=len(buckets), bucket_elems=args.bucket_elems,
                                                backward="one fp16 GEMM [L/768,k]x[k,768] per bucket "
                                                         f"per rank, k={k}",
                                                step_stream_priority=args.step_priority,
                                                step_sms=args.step_sms or "all",
                                                gemm_carveout_sms=carve),
            "backward_ms": t_b, "backward_carved_ms": t_b_carved, "step_ms": t_s, "serial_ms": t_serial, "overlapped_ms": t_over,
            "gpu_launches_per_rep": len(buckets) * (P + 1),
        }
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def run_offload(args, wl, mode, dist):
    """ZeRO-Offload step: fp16 gradient mean to page-locked host memory, CPU
    Adam per piece of shards as its gradients arrive, fp16 weights back into
    the device vector while the next piece is updated.  Also timed alone:
    the GPU reduce (its host writes) and the host Adam on all host cores."""
    import torch

    import zero_sharded_mixed_shard_gb300 as z
    from zero_sharded_mixed_shard_gb300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the fused step has no CPU path)")
    if wl.shard is not None:
        raise SystemExit("--offload runs whole-vector workloads")
    torch.cuda.set_device(dist.local_rank)
    dist.init("nccl")
    dev = torch.device("cuda", dist.local_rank)
    P, N = wl.P, wl.N
    stride = wl.rank_stride(True)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    g = synth.torch_grads(P, N, stride, wl.grad_sigma, wl.seed, dev, wl.heavy_tail_frac,
                          wl.zero_frac, step=1)
    dstate = synth.torch_state(N, wl.seed, dev, wl.master_sigma)
    host = [torch.empty(N, dtype=torch.float32, pin_memory=True) for _ in range(3)]
    for h, d in zip(host, dstate[:3]):
        h.copy_(d)
    g16_h = torch.empty(N, dtype=torch.float16, pin_memory=True)
    p16_h = torch.empty(N, dtype=torch.float16, pin_memory=True)
    params = dstate[3]
    stream = torch.cuda.current_stream(dev)
    t = [0]

    def step():
        t[0] += 1
        z.zero_offload_step(g, stride, *host, g16_h, p16_h, params, N, P, wl.stage, t[0], wl.lr,
                            wl.b1, wl.b2, wl.eps, mode, 0, stream)

    def reduce_only():
        z.zero_reduce_scatter_fp16(g, stride, 0, P, N, g16_h, stream)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return dist.max(e0.elapsed_time(e1) / reps, dev)

    reps = max(3, min(args.steps, 20))
    ms_step = timed(step, reps)
    ms_reduce = timed(reduce_only, reps)
    # the host update alone, all cores, same buffers
    t0 = time.perf_counter()
    for k in range(reps):
        z.zero_cpu_adam(g16_h, *host, p16_h, N, t[0] + k + 1, wl.lr, wl.b1, wl.b2, wl.eps, mode, 0)
    ms_cpu = (time.perf_counter() - t0) * 1e3 / reps
    if dist.rank == 0:
        line = {
            "metric": "params updated/sec, ZeRO-Offload step (update on the host CPU)",
            "value": N * dist.world / (ms_step / 1e3), "unit": "params/s", "n_gpus": dist.world,
            "steps": reps, "warmup": 3, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "dtype": "f32", "data": "synthetic (seeded device RNG)",
            "config": dict(workload_config(wl, mode), state="fp32 master/m/v in page-locked host memory"),
            "reduce_ms": ms_reduce,
            "reduce_gbs": (2 * P + 2) * N / (ms_reduce / 1e3) / 1e9,
            "cpu_adam_ms": ms_cpu, "cpu_adam_params_per_s": N / (ms_cpu / 1e3), "cpu_cores": cores,
            "cpu_adam_host_gbs": 28 * N / (ms_cpu / 1e3) / 1e9,
            "host_link_bytes_per_step": {"d2h_fp16_gradient": 2 * N, "h2d_fp16_params": 2 * N},
            "device_state_bytes_saved": 12 * N,
        }
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def run_mlp4(args, dist):
    """Training steps of the 4-layer scalar MLP on 4 simulated ranks (one
    layer each), layer-pipelined on two streams and serial on one."""
    import numpy as np
    import torch

    import zero_sharded_mixed_shard_gb300 as z

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(dist.local_rank)
    dist.init("nccl")
    P, n = 4, 256
    rng = np.random.default_rng(0)
    dev = torch.device("cuda", dist.local_rank)
    master0 = torch.tensor([rng.uniform(0.6, 1.2) if i % 2 == 0 else rng.uniform(0.0, 0.2)
                            for i in range(8)], dtype=torch.float32, device=dev)
    x = torch.from_numpy(rng.uniform(0.1, 1.0, (P, n)).astype(np.float32)).to(dev)
    main, side = torch.cuda.current_stream(dev), torch.cuda.Stream(dev)
    reps = max(10, min(args.steps, 2000))
    out = {}
    for pipelined in (True, False):
        master, m, v = master0.clone(), torch.zeros(8, device=dev), torch.zeros(8, device=dev)
        shard16 = master0.half()
        gathered16 = torch.zeros(8, dtype=torch.float16, device=dev)
        grads16 = torch.zeros((P, 8), dtype=torch.float16, device=dev)
        loss = torch.zeros(P, device=dev)
        t = 0

        def step():
            nonlocal t
            t += 1
            z.zero_mlp4_zero3_step(x, P, n, gathered16, master, m, v, shard16, grads16, 8, loss, t,
                                   1e-2, 0.9, 0.999, 1e-8, 0, pipelined=pipelined,
                                   main_stream=main, step_stream=side)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        loss0 = float(loss.mean())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        e0.record(main)
        for _ in range(reps):
            step()
        e1.record(main)
        host_us = (time.perf_counter() - h0) * 1e6 / reps   # enqueueing only: before the wait
        torch.cuda.synchronize()
        out["pipelined" if pipelined else "serial"] = {
            "us_per_step": e0.elapsed_time(e1) * 1e3 / reps, "host_enqueue_us_per_step": host_us,
            "loss_after_warmup": loss0, "loss_at_end": float(loss.mean())}
    if dist.rank == 0:
        line = {"metric": "microseconds per training step, layer-pipelined ZeRO-3 (4-layer scalar MLP)",
                "value": out["pipelined"]["us_per_step"], "unit": "us/step", "n_gpus": dist.world,
                "steps": reps, "warmup": args.warmup, "higher_is_better": False, "dtype": "f32",
                "data": "synthetic", "config": {"workload": f"mlp4: P={P} ranks, {n} samples each, "
                                                            "one layer (w, b) per rank"},
                "gpu_launches_per_step": 1 + 4 + 4 + 1, **out}
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def main(argv=None):
    args = parse_args(argv)
    from zero_sharded_mixed_shard_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.ranks is not None:
        if wl.shard is not None or not 1 <= args.ranks <= 1024:
            raise SystemExit("--ranks takes 1..1024 on a whole-vector workload")
        wl = dataclasses.replace(wl, P=args.ranks, name=f"{wl.name}-P{args.ranks}")
    if args.elements is not None:
        if wl.shard is not None or args.elements < 1:
            raise SystemExit("--elements takes N >= 1 on a whole-vector workload")
        wl = dataclasses.replace(wl, N=args.elements, tensors=None, name=f"{wl.name}-N{args.elements}")
    mode = wl.modes[0] if args.mode is None else args.mode
    dist = Dist()
    if args.gpus != dist.world:
        raise SystemExit(f"--gpus {args.gpus} but {dist.world} process(es): launch N > 1 as "
                         f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}")
    if args.impl == "reference":
        return run_reference(args, wl, mode, dist)
    if args.overlap:
        return run_overlap(args, wl, mode, dist)
    if args.offload:
        return run_offload(args, wl, mode, dist)
    if args.mlp4:
        return run_mlp4(args, dist)
    return run_ours(args, wl, mode, dist)


if __name__ == "__main__":
    sys.exit(main())
