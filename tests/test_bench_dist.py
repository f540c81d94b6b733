"""The multi-rank host logic of bench.py on two CPU ranks (gloo): each rank gets its own batch,
the job time is the slowest rank's, and the whole-job throughput counts every rank's work.
The reference arm runs on rank 0 only.  No GPU is needed."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    from frame_aligned_block_fsa_b300.inputs import make_qkv
    from frame_aligned_block_fsa_b300.workloads import WORKLOADS

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        wl = WORKLOADS["tiny"]
        seed = bench.rank_seed(wl, rank)
        q, _, _ = make_qkv(wl.H, wl.N, wl.D, seed=seed, kind=wl.kind)
        # every rank times its own steps; rank 1 is the slow one here
        own_ms = 10.0 + 5.0 * rank
        job_ms = bench.max_over_ranks(own_ms, dist, torch.device("cpu"))
        value = bench.job_throughput(1e12, world, 4, job_ms)

        class Args:
            workload = "tiny"
            steps = 1
            warmup = 0
        ref = bench.reference_arm(Args(), rank) if rank != 0 else "skipped"
        dist.barrier()
        results[rank] = (seed, float(q.float().sum()), job_ms, value, ref)
    finally:
        dist.destroy_process_group()


def test_two_ranks_weak_scaling_host_logic():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    (s0, q0, t0, v0, r0), (s1, q1, t1, v1, r1) = res[0], res[1]
    assert s0 != s1 and q0 != q1          # independent batches of the same shape
    assert t0 == t1 == 15.0               # the slowest rank's time, seen by every rank
    assert v0 == v1 == pytest.approx(1e12 * 2 * 4 / 15e-3 / 1e12)
    assert r1 is None                     # the reference arm does no work off rank 0


def test_reference_arm_prints_the_contract_line():
    # bench.py --impl reference runs the oracle on host cores: one JSON line with the keys of
    # the bench contract, the cpu_baseline describing this run and a zero-copy e2e
    import json
    import subprocess

    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny", "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
