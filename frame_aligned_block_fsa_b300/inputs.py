"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers; it holds none of the attention arithmetic.

Recipes (the pages measure on production data, which is not available):
  normal: Q, K, V i.i.d. N(0, 1), rounded to bf16, layout [H][N][D].
  stress: every Q and K row is N(0, I_D) times an independent LogNormal(0, 1)
          scalar (per head, per token); in each head ceil(0.001 N) key tokens,
          chosen uniformly without replacement, are further scaled by 8;
          V is N(0, 1).
  offset: as normal, then one vector m_h ~ N(0, 4^2 I_D) per head is added to every key
          of head h (a large component that all keys share).
  loose:  as normal, then the keys of head h are scaled by 3 + 0.5 (h mod 4): the logits
          spread out, and the norm bound sits 20 to 60 nats above the row max while the head
          still passes the gap test at a raised tau (a loose but eligible bound).
  prep:   hidden states x ~ N(0, 1) [N][d_model] and projection weights
          w ~ N(0, 1/d_model) [3 H D][d_model], drawn in that order (make_prep_inputs).
All draws come from one CPU torch.Generator seeded with the workload's seed, in
the order q, k, v (then the stress scalars and outlier choice, or the key offsets), so a seed fixes
the inputs on every machine.
"""
from __future__ import annotations

import math

import torch

from .workloads import Workload


KEY_OFFSET_STD = 4.0  # spread of the shared key component of the "offset" inputs


def make_qkv(H: int, N: int, D: int, seed: int, kind: str = "normal"):
    """Return (q, k, v) as contiguous CPU bf16 tensors of shape [H, N, D]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((H, N, D), generator=g, dtype=torch.float32)
    k = torch.randn((H, N, D), generator=g, dtype=torch.float32)
    v = torch.randn((H, N, D), generator=g, dtype=torch.float32)
    if kind == "stress":
        qs = torch.randn((H, N, 1), generator=g, dtype=torch.float32).exp_()
        ks = torch.randn((H, N, 1), generator=g, dtype=torch.float32).exp_()
        q.mul_(qs)
        k.mul_(ks)
        n_out = math.ceil(0.001 * N)
        for h in range(H):
            idx = torch.randperm(N, generator=g)[:n_out]
            k[h, idx, :] *= 8.0
    elif kind == "offset":
        m = torch.randn((H, 1, D), generator=g, dtype=torch.float32).mul_(KEY_OFFSET_STD)
        k.add_(m)
    elif kind == "loose":
        scale = torch.tensor([3.0 + 0.5 * (h % 4) for h in range(H)], dtype=torch.float32).view(H, 1, 1)
        k.mul_(scale)
    elif kind != "normal":
        raise ValueError(f"unknown input kind {kind!r}")
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_prep_inputs(N: int, d_model: int, H: int, D: int, seed: int):
    """Hidden states x ~ N(0, 1) [N][d_model] and projection weights w ~ N(0, 1/d_model)
    [3 H D][d_model] (q, k, v rows, head-major), both bf16 on the CPU; with unit-RMS rows after
    the normalisation, q, k and v come out about N(0, 1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn((N, d_model), generator=g, dtype=torch.float32)
    w = torch.randn((3 * H * D, d_model), generator=g, dtype=torch.float32).mul_(1.0 / math.sqrt(d_model))
    return x.to(torch.bfloat16).contiguous(), w.to(torch.bfloat16).contiguous()


def make_workload_inputs(wl: Workload):
    return make_qkv(wl.H, wl.N, wl.D, wl.seed, wl.kind)


def sample_rows(wl: Workload, per_head: int, seed: int = 12345):
    """Stratified row sample: every frame, first/last row of every 16-row group edge
    that matters (frame starts/ends, 128-row tile edges, the ragged tail of each
    frame), topped up with uniform random rows.  Returns (heads int32[R], rows int64[R])."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    heads, rows = [], []
    F, T, N = wl.F, wl.T, wl.N
    special = set()
    for f in range(F):
        base = f * T
        special.update({base, base + T - 1})
        for t0 in range(0, T, 128):
            special.update({base + t0, base + min(t0 + 127, T - 1)})
    special = sorted(special)
    for h in range(wl.H):
        pick = list(special)
        if len(pick) > per_head:
            idx = torch.randperm(len(pick), generator=g)[:per_head].tolist()
            pick = [pick[i] for i in sorted(idx)]
        extra = per_head - len(pick)
        if extra > 0:
            pick += torch.randint(0, N, (extra,), generator=g).tolist()
        heads += [h] * len(pick)
        rows += pick
    import numpy as np

    return np.asarray(heads, dtype=np.int32), np.asarray(rows, dtype=np.int64)
