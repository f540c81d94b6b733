#!/usr/bin/env python
"""Benchmark: frame-aligned sparse attention (norm-bound softmax) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step = the whole hot path over one batch held in HBM: fsa_norms (per-row norms,
per-frame max key norms, row bounds, per-head eligibility) followed by the attention
kernel, for every head of the 28.8k-token workload (F=24 frames x T=1200 tokens, H=24,
D=128, window +-2 frames plus reference frame 0, block 80).  Metric: effective TFLOPS over
active-block FLOPs, 4 D T^2 sum_f |S(f)| H per step (QK^T and PV over active frame pairs;
no padding rows, no softmax FLOPs).  Prints one JSON line.

Under torchrun each rank processes its own independent batch (same shape, its own seed):
no collective touches the data path; barriers and a max-reduction of the timings only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn effective TFLOPS (active blocks) & % of B300 bf16 tensor peak"
UNIT = "TFLOPS"
WORKLOAD = "sr28k"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_sr28k_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "frame_aligned_block_fsa_b300", "csrc", f)
                  for f in ("fsa_attn.cu", "fsa_ptx.cuh", "fsa_internal.h")]
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["fsa", "reference"], default="fsa")
    ap.add_argument("--mode", choices=["norm_bound", "online_max"], default="norm_bound")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--center-keys", action="store_true", help="mean-centred key norms in the bound")
    ap.add_argument("--prep", action="store_true",
                    help="step = fsa_prep (hidden states -> q, k, v and norms) + attention")
    ap.add_argument("--d-model", type=int, default=0, help="prep model width (default H*D)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU-baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-extras", action="store_true", help="skip the online-max comparison and gap stats")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: one JSON line per workload and softmax mode (attention time, "
                         "norms time, bound-gap statistics, fallback heads, underflow rows)")
    ap.add_argument("--sweep-part", choices=["all", "workloads", "key_tile", "masked"], default="all",
                    help="with --sweep: every part, or only the workload/mode lines, the key-tile sweep, or the "
                         "masked-block comparison")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(wl, rank: int) -> int:
    """Seed of a rank's inputs: every rank gets its own independent batch of the workload."""
    return wl.seed + 1000 * rank


def max_over_ranks(value: float, pg, device) -> float:
    """The largest of the ranks' values (the whole job ends when its slowest rank does)."""
    if pg is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, world: int, steps: int, ms: float) -> float:
    """Whole-job TFLOP/s: the active FLOPs of every rank's steps over the slowest rank's time."""
    return flops_per_rank_step * world * steps / (ms * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic():
    """DRAM bytes per attention launch from the committed ncu summary, if it matches this kernel."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as fh:
        d = json.load(fh)
    if d.get("kernel_sha") != kernel_hash():
        return None
    return d.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile

        fd, self.path = tempfile.mkstemp(prefix="fsa_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        loaded = [s for s in sm if mx and s >= 0.3 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def cpu_oracle_leg(wl, target_seconds: float, seed_rows: int = 7):
    """Time the fp64 oracle on a bounded row sample of the workload (host cores)."""
    import numpy as np

    import oracle
    from frame_aligned_block_fsa_b300.inputs import make_workload_inputs

    q, k, v = make_workload_inputs(wl)
    threads = oracle.default_threads()
    rng = np.random.default_rng(seed_rows)

    def run(n):
        heads = rng.integers(0, wl.H, n).astype(np.int32)
        rows = rng.integers(0, wl.N, n).astype(np.int64)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, wl.F, wl.T, wl.w, wl.ref, heads, rows, nthreads=threads)
        dt = time.perf_counter() - t0
        frames = rows // wl.T
        flops = sum(4 * wl.D * wl.T * oracle.frame_set_size(wl.F, wl.w, wl.ref, int(f)) for f in frames)
        return n, dt, flops

    run(threads)  # warm-up: thread start-up and first touch of the inputs
    # batches of rows until about target_seconds of oracle time have been measured
    n, dt, flops, batch = 0, 0.0, 0, 64 * threads
    while dt < target_seconds:
        bn, bdt, bfl = run(batch)
        n, dt, flops = n + bn, dt + bdt, flops + bfl
        if bdt < 0.25 * target_seconds:
            batch *= 2
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} random rows of {wl.name} (all heads), fp64 dense masked attention over all "
                      f"{wl.N} keys per row, {dt:.1f} s"}


def reference_arm(args, rank):
    """--impl reference: the fp64 oracle on host cores, one bounded row sample per step."""
    from frame_aligned_block_fsa_b300.workloads import WORKLOADS

    if rank != 0:
        return
    import numpy as np

    import oracle
    from frame_aligned_block_fsa_b300.inputs import make_workload_inputs

    wl = WORKLOADS[args.workload]
    q, k, v = make_workload_inputs(wl)
    threads = oracle.default_threads()
    rng = np.random.default_rng(11)
    rows_per_step = 4 * threads

    def step():
        heads = rng.integers(0, wl.H, rows_per_step).astype(np.int32)
        rows = rng.integers(0, wl.N, rows_per_step).astype(np.int64)
        oracle.attention_rows(q, k, v, wl.F, wl.T, wl.w, wl.ref, heads, rows, nthreads=threads)
        return sum(4 * wl.D * wl.T * oracle.frame_set_size(wl.F, wl.w, wl.ref, int(r // wl.T)) for r in rows)

    for _ in range(args.warmup):
        step()
    flops = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flops += step()
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": workload_desc(wl), "mode": "dense fp64 masked attention (oracle)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{rows_per_step} random rows per step of {wl.name}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _timed(fn, reps, stream):
    """Mean milliseconds of `reps` calls of fn after three untimed ones (CUDA events on `stream`)."""
    import torch

    for _ in range(3):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def sweep(args):
    """One JSON line per measurement (not the bench contract line):
    workloads -- every workload in both softmax modes, and in norm_bound mode once more with
                 mean-centred keys;
    key_tile  -- the attention kernel at key tiles of 16, 32, 48, 64, 96 and 128 keys, both modes, at the
                 28.8k and 57.6k workloads (the block geometry retuned for the softmax);
    masked    -- the masked-block comparison variant at blocks of 128, 256 and 512 tokens beside
                 the frame-aligned kernel in both modes, at the 28.8k, 57.6k and stress workloads."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.sweep_part in ("all", "workloads"):
        sweep_workloads(args, dev)
    if args.sweep_part in ("all", "key_tile"):
        sweep_key_tile(args, dev)
    if args.sweep_part in ("all", "masked"):
        sweep_masked(args, dev)


def sweep_key_tile(args, dev):
    import torch

    import frame_aligned_block_fsa_b300 as fsa
    from frame_aligned_block_fsa_b300.inputs import make_workload_inputs
    from frame_aligned_block_fsa_b300.workloads import WORKLOADS

    stream = torch.cuda.current_stream()
    peaks, _ = load_peaks()
    reps = max(3, min(args.steps, 20))
    for name in ("sr28k", "sr57k"):
        wl = WORKLOADS[name]
        q, k, v = (t.to(dev) for t in make_workload_inputs(wl))
        H, N, D = wl.H, wl.N, wl.D
        out = torch.empty((H, N, D), dtype=torch.float32, device=dev)
        lse = torch.empty((H, N), dtype=torch.float32, device=dev)
        bound = torch.empty((H, N), dtype=torch.float32, device=dev)
        elig = torch.empty(H, dtype=torch.uint8, device=dev)
        with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
            flops = plan.nnz() * 4 * wl.block * wl.block * D * H
            fsa.norms(q, k, plan, None, None, bound, elig, stream=stream)
            for key_tile in (16, 32, 48, 64, 96, 128):
                plan.set_key_tile(key_tile)
                for mode in ("norm_bound", "online_max"):
                    ms = _timed(lambda: fsa.forward_ex(q, k, v, plan, mode, out=out, lse=lse, bound=bound,
                                                       eligible=elig, stream=stream), reps, stream)
                    tf = flops / (ms * 1e-3) / 1e12
                    print(json.dumps({"sweep": name, "part": "key_tile", "key_tile": key_tile, "mode": mode,
                                      "workload": workload_desc(wl), "attention_ms": ms, "attention_tflops": tf,
                                      "frac_of_bf16_peak": tf / float(peaks["bf16_tflops"])}), flush=True)
        del q, k, v, out, lse, bound, elig
        torch.cuda.empty_cache()


def sweep_masked(args, dev):
    import torch

    import frame_aligned_block_fsa_b300 as fsa
    from frame_aligned_block_fsa_b300.inputs import make_workload_inputs
    from frame_aligned_block_fsa_b300.workloads import WORKLOADS

    stream = torch.cuda.current_stream()
    peaks, _ = load_peaks()
    reps = max(3, min(args.steps, 20))
    for name in ("sr28k", "sr57k", "stress"):
        wl = WORKLOADS[name]
        q, k, v = (t.to(dev) for t in make_workload_inputs(wl))
        H, N, D = wl.H, wl.N, wl.D
        out = torch.empty((H, N, D), dtype=torch.float32, device=dev)
        lse = torch.empty((H, N), dtype=torch.float32, device=dev)
        bound = torch.empty((H, N), dtype=torch.float32, device=dev)
        elig = torch.empty(H, dtype=torch.uint8, device=dev)
        with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
            active_pairs = plan.nnz() * wl.block * wl.block * H
            flops = 4 * active_pairs * D
            norms_ms = _timed(lambda: fsa.norms(q, k, plan, None, None, bound, elig, stream=stream), reps, stream)
            base = {}
            for mode in ("norm_bound", "online_max"):
                base[mode] = _timed(lambda: fsa.forward_ex(q, k, v, plan, mode, out=out, lse=lse, bound=bound,
                                                           eligible=elig, stream=stream), reps, stream)
            for block in (128, 256, 512):
                st = fsa.new_stats(dev)
                fsa.forward_masked(q, k, v, plan, block=block, out=out, lse=lse, stats=st)
                torch.cuda.synchronize()
                stats = fsa.read_stats(st)
                ms = _timed(lambda: fsa.forward_masked(q, k, v, plan, block=block, out=out, lse=lse, stream=stream),
                            reps, stream)
                tf = flops / (ms * 1e-3) / 1e12
                print(json.dumps({
                    "sweep": name, "part": "masked", "block": block, "workload": workload_desc(wl),
                    "masked_ms": ms, "masked_tflops_active": tf, "frac_of_bf16_peak": tf / float(peaks["bf16_tflops"]),
                    "computed_pairs_over_active": stats["pairs_visited"] / active_pairs,
                    "frame_aligned_online_ms": base["online_max"], "frame_aligned_norm_bound_ms": base["norm_bound"],
                    "norms_ms": norms_ms,
                    # masked time over frame-aligned time (> 1: the frame-aligned layout is faster)
                    "speedup_frame_aligned_online": ms / base["online_max"],
                    "speedup_frame_aligned_norm_bound_incl_norms": ms / (base["norm_bound"] + norms_ms),
                    "error": stats["error"]}), flush=True)
        del q, k, v, out, lse, bound, elig
        torch.cuda.empty_cache()


def sweep_workloads(args, dev):
    import torch

    import frame_aligned_block_fsa_b300 as fsa
    from frame_aligned_block_fsa_b300.inputs import make_workload_inputs
    from frame_aligned_block_fsa_b300.workloads import WORKLOADS

    stream = torch.cuda.current_stream()
    peaks, _ = load_peaks()
    cached = {}  # the current workload's device inputs, shared by its two centring settings
    for name, center in [(n, c) for n in ("tiny", "small", "sr28k", "sr57k", "stress", "offset")
                         for c in (False, True)]:
        wl = WORKLOADS[name]
        if cached.get("name") != name:
            cached.clear()
            torch.cuda.empty_cache()
            cached.update(name=name, qkv=tuple(t.to(dev) for t in make_workload_inputs(wl)))
        q, k, v = cached["qkv"]
        H, N, D = wl.H, wl.N, wl.D
        out = torch.empty((H, N, D), dtype=torch.float32, device=dev)
        lse = torch.empty((H, N), dtype=torch.float32, device=dev)
        bound = torch.empty((H, N), dtype=torch.float32, device=dev)
        elig = torch.empty(H, dtype=torch.uint8, device=dev)
        rm = torch.empty((H, N), dtype=torch.float32, device=dev)
        plan = fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block)
        plan.set_center_keys(center)
        flops = plan.nnz() * 4 * wl.block * wl.block * D * H
        reps = max(3, min(args.steps, 20))

        def timed(fn):
            return _timed(fn, reps, stream)

        norms_ms = timed(lambda: fsa.norms(q, k, plan, None, None, bound, elig, stream=stream))
        # the row max comes from a running-max pass over every head
        fsa.forward_ex(q, k, v, plan, "online_max", out=out, lse=lse, bound=bound, eligible=elig, rowmax=rm)
        torch.cuda.synchronize()
        gap = (bound - rm).flatten()
        qs = torch.quantile(gap[torch.randperm(gap.numel(), device=dev)[:1 << 20]],
                            torch.tensor([0.5, 0.99], device=dev))
        for mode in ("norm_bound",) if center else ("norm_bound", "online_max"):
            st = fsa.new_stats(dev)
            fsa.forward_ex(q, k, v, plan, mode, out=out, lse=lse, bound=bound, eligible=elig, stats=st)
            torch.cuda.synchronize()
            stats = fsa.read_stats(st)
            ms = timed(lambda: fsa.forward_ex(q, k, v, plan, mode, out=out, lse=lse, bound=bound, eligible=elig,
                                              stream=stream))
            line = {"sweep": name, "mode": mode, "center_keys": center, "workload": workload_desc(wl),
                    "attention_ms": ms,
                    "attention_tflops": flops / (ms * 1e-3) / 1e12,
                    "frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / float(peaks["bf16_tflops"]),
                    "norms_ms": norms_ms, "active_flops": flops, "eligible_heads": int(elig.sum().item()),
                    "heads": H, "fallback_heads": stats["fallback_heads"], "underflow_rows": stats["underflow_rows"],
                    "error": stats["error"],
                    "bound_gap_nats": {"min": float(gap.min()), "median": float(qs[0]), "p99": float(qs[1]),
                                       "max": float(gap.max())}}
            print(json.dumps(line), flush=True)
        plan.close()
        del q, k, v, out, lse, bound, elig, rm
        torch.cuda.empty_cache()


def workload_desc(wl):
    return (f"{wl.name}: F={wl.F} x T={wl.T} (N={wl.N}), H={wl.H}, D={wl.D}, window +-{wl.w} + ref frame "
            f"{wl.ref}, block {wl.block}, inputs {wl.kind}, seed {wl.seed}")


def main():
    args = parse()
    rank, world, local = dist_info()
    if args.impl == "reference":
        return reference_arm(args, rank)
    if args.sweep:
        return sweep(args) if rank == 0 else None

    import numpy as np
    import torch

    import frame_aligned_block_fsa_b300 as fsa
    from frame_aligned_block_fsa_b300.inputs import make_prep_inputs, make_qkv
    from frame_aligned_block_fsa_b300.workloads import WORKLOADS

    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    wl = WORKLOADS[args.workload]
    H, N, D = wl.H, wl.N, wl.D
    # each rank: its own independent batch of the same shape
    q_h, k_h, v_h = make_qkv(H, N, D, seed=rank_seed(wl, rank), kind=wl.kind)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    out = torch.empty((H, N, D), dtype=torch.float32, device=dev)
    lse = torch.empty((H, N), dtype=torch.float32, device=dev)
    bound = torch.empty((H, N), dtype=torch.float32, device=dev)
    elig = torch.empty(H, dtype=torch.uint8, device=dev)
    plan = fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block)
    plan.set_center_keys(args.center_keys)
    # active FLOPs: every active (query block, key block) pair does QK^T and PV, 2 * 2 B^2 D each
    flops_step = plan.nnz() * 4 * wl.block * wl.block * D * H
    stream = torch.cuda.current_stream()
    if args.prep:
        # hidden states and projection weights of d_model = H * D; q, k, v are overwritten by
        # the prep every step
        dm = args.d_model or H * D
        x, w = (t.to(dev) for t in make_prep_inputs(N, dm, H, D, seed=rank_seed(wl, rank) + 1000))
        prep_flops = 2 * N * dm * 3 * H * D

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if args.prep:
            fsa.prep(x, w, plan, H, q=q, k=k, v=v, bound=bound, eligible=elig, stream=stream)
        else:
            fsa.norms(q, k, plan, None, None, bound, elig, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        fsa.forward_ex(q, k, v, plan, args.mode, out=out, lse=lse, bound=bound, eligible=elig, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step()
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    norms_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = max_over_ranks(total_ms, pg, dev)
    ms_step = total_ms / args.steps
    value = job_throughput(flops_step, world, args.steps, total_ms)

    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if not args.no_e2e and not args.prep:
        # fsa_forward_host: pinned host q, k, v in, pinned host out, lse back; the library
        # pipelines chunks of heads over copy-in, compute and copy-out streams
        qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        out_h = torch.empty((H, N, D), dtype=torch.float32).pin_memory()
        lse_h = torch.empty((H, N), dtype=torch.float32).pin_memory()
        e2e_steps = max(3, min(args.steps, 10))

        def e2e_step():
            fsa.forward_host(qp, kp, vp, plan, args.mode, out=out_h, lse=lse_h, stream=stream)

        for _ in range(2):
            e2e_step()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        barrier()
        e2e_ms = a.elapsed_time(b)
        e2e_ms = max_over_ranks(e2e_ms, pg, dev)
        e2e = {"value": job_throughput(flops_step, world, e2e_steps, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": 3 * H * N * D * 2, "d2h_bytes_per_step": H * N * D * 4 + H * N * 4,
               "ms_per_step": e2e_ms / e2e_steps,
               "path": "fsa_forward_host: pinned host q,k,v -> chunks of heads copied in, normed and attended, "
                       "copied out on three streams -> pinned host out, lse"}

    # ---------------------------------------------------------------- comparison / diagnostics
    extras = {}
    if not args.no_extras:
        st = fsa.new_stats(dev)
        rm = torch.empty((H, N), dtype=torch.float32, device=dev)
        fsa.forward_ex(q, k, v, plan, "norm_bound", out=out, lse=lse, bound=bound, eligible=elig, stats=st)
        torch.cuda.synchronize()
        s_nb = fsa.read_stats(st)
        # online-max comparison point: same kernel, running max on every head
        other = "online_max" if args.mode == "norm_bound" else "norm_bound"
        for _ in range(3):
            fsa.forward_ex(q, k, v, plan, other, out=out, lse=lse, bound=bound, eligible=elig)
        oe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        reps = max(5, args.steps // 2)
        torch.cuda.synchronize()
        oe[0].record(stream)
        for _ in range(reps):
            fsa.forward_ex(q, k, v, plan, other, out=out, lse=lse, bound=bound, eligible=elig)
        oe[1].record(stream)
        torch.cuda.synchronize()
        other_ms = oe[0].elapsed_time(oe[1]) / reps
        fsa.forward_ex(q, k, v, plan, "online_max", out=out, lse=lse, bound=bound, eligible=elig, rowmax=rm)
        torch.cuda.synchronize()
        gap = (bound - rm).flatten()
        qs = torch.quantile(gap[torch.randperm(gap.numel(), device=dev)[:1 << 20]],
                            torch.tensor([0.5, 0.99], device=dev))
        # Sustained: the attention kernel back to back for about a second, the regime of the
        # measured sustained GEMM peak (the power cap lowers the clock after ~0.1 s of load);
        # every tenth launch is timed, and the last half of them gives the median.
        sus_ms = []
        se = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        t_sus = time.time()
        while time.time() - t_sus < 1.0 or len(sus_ms) < 20:
            se[0].record(stream)
            fsa.forward_ex(q, k, v, plan, args.mode, out=out, lse=lse, bound=bound, eligible=elig, stream=stream)
            se[1].record(stream)
            for _ in range(9):
                fsa.forward_ex(q, k, v, plan, args.mode, out=out, lse=lse, bound=bound, eligible=elig,
                               stream=stream)
            torch.cuda.synchronize()
            sus_ms.append(se[0].elapsed_time(se[1]))
        sus_med = statistics.median(sus_ms[len(sus_ms) // 2:])
        extras = {
            "sustained": {"attention_ms_median": sus_med, "launches": 10 * len(sus_ms),
                          "seconds": time.time() - t_sus,
                          "achieved": flops_step / (sus_med * 1e-3) / 1e12},
            f"attention_ms_{args.mode}": statistics.median(attn_ms),
            f"attention_ms_{other}": other_ms,
            f"attention_tflops_{other}": flops_step / (other_ms * 1e-3) / 1e12,
            "bound_gap_nats": {"min": float(gap.min()), "median": float(qs[0]), "p99": float(qs[1]),
                               "max": float(gap.max())},
            "eligible_heads": int(elig.sum().item()), "heads": H,
            "fallback_heads": s_nb["fallback_heads"], "underflow_rows": s_nb["underflow_rows"],
        }

    peaks, peak_src = load_peaks()
    attn_med = statistics.median(attn_ms)
    attn_avg = sum(attn_ms) / len(attn_ms)
    achieved = flops_step / (attn_avg * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    # Q and K read once, bound written, per-frame key statistics; centring reads K once more
    norms_bytes = (3 if args.center_keys else 2) * H * N * D * 2 + 4 * H * N + 4 * H * wl.F * (D + 1) + H
    norms_avg = sum(norms_ms) / len(norms_ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(wl), "mode": args.mode, "center_keys": args.center_keys,
                   "step": (f"fsa_prep (x [N, {dm}] -> q, k, v, norms) + attention, all heads" if args.prep
                            else "fsa_norms + attention, all heads"),
                   "l2": f"inputs {3 * H * N * D * 2 / 1e6:.0f} MB > 126 MB L2, no flush",
                   "active_flops_per_step": flops_step, "parallelism": f"independent batch per rank x{world}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": load_traffic(),
                     "kernel": f"fsa_attn_fwd_kernel<{D}> (persistent)", "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "attention_ms_avg": attn_avg, "attention_ms_median": attn_med,
                     "attention_ms_min": min(attn_ms), "attention_ms_first": attn_ms[0],
                     "attention_ms_last": attn_ms[-1]},
        "norms_roofline": {"bound": "hbm", "achieved": norms_bytes / (norms_avg * 1e-3) / 1e9,
                           "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                           "frac": norms_bytes / (norms_avg * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                           "ms_avg": norms_avg, "algorithmic_bytes": norms_bytes},
        "clocks": clk,
        # per step: 2 norm kernels (3 with centred keys), or the prep's 6 (rms, K/V projection,
        # frame key sums, key-set statistics, Q projection, eligibility), + the attention kernel
        "gpu_launches": (7 if args.prep else (4 if args.center_keys else 3)) * args.steps,
        "e2e": e2e,
    }
    sus = extras.pop("sustained", None)
    line.update(extras)
    if sus is not None:
        # the same kernel under sustained load, against the sustained GEMM peak
        sp = float(peaks.get("bf16_tflops_sustained", peak))
        line["roofline"]["sustained"] = {"achieved": sus["achieved"], "peak": sp, "frac": sus["achieved"] / sp,
                                         "attention_ms_median": sus["attention_ms_median"],
                                         "launches": sus["launches"], "seconds": sus["seconds"],
                                         "peak_source": f"{peak_src} bf16_tflops_sustained"}
    if args.prep:
        prep_avg = norms_avg
        line.pop("norms_roofline")
        line["prep_roofline"] = {"bound": "tensor", "achieved": prep_flops / (prep_avg * 1e-3) / 1e12,
                                 "peak": peak, "unit": "TFLOP/s",
                                 "frac": prep_flops / (prep_avg * 1e-3) / 1e12 / peak, "ms_avg": prep_avg,
                                 "flops": prep_flops,
                                 "kernel": "rms_kernel + fsa_prep_kernel (one cooperative launch) + eligibility"}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_leg(wl, target_seconds=12.0)
    plan.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
