"""GPU parity of the masked block variant (fsa_forward_masked) against the fp64 oracle.

The variant computes the same attention as the frame-aligned path, the way a general
block-sparse kernel with a mask would: blocks of a multiple of 128 tokens over the padded
sequence, mask predicates on the tiles a frame boundary cuts, the window and the reference frame
as two passes and a merge.  Its results are held to the unit-variance tolerance of the
frame-aligned path (max-abs 1e-2, mean-abs 1e-3 on out and lse): both passes run the same
running-max softmax with bf16 weights and fp32 accumulation, and the merge adds one fp32
rescale per element.
"""
import numpy as np
import pytest
import torch

import frame_aligned_block_fsa_b300 as fsa
from frame_aligned_block_fsa_b300.inputs import make_qkv, make_workload_inputs, sample_rows
from frame_aligned_block_fsa_b300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3

_cache = {}


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from frame_aligned_block_fsa_b300 import build

    build.build()
    fsa.load()
    return torch.device("cuda:0")


def _inputs(name):
    if name not in _cache:
        _cache[name] = make_workload_inputs(WORKLOADS[name])
    return _cache[name]


def _masked(dev, q, k, v, F, T, w, ref, block, stats=False):
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    st = fsa.new_stats(dev) if stats else None
    # the plan's own block size is not used by the masked variant; 16 divides every T here
    with fsa.Plan(F, T, w, ref, 16) as plan:
        out, lse = fsa.forward_masked(qd, kd, vd, plan, block=block, stats=st)
        torch.cuda.synchronize()
    res = {"out": out.cpu().double().numpy(), "lse": lse.cpu().double().numpy()}
    if stats:
        res["stats"] = fsa.read_stats(st)
        assert res["stats"]["error"] == 0, res["stats"]
    return res


def _check(out, lse, ref_out, ref_lse):
    d = np.abs(out - ref_out)
    dl = np.abs(lse - ref_lse)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert d.max() <= MAX_ABS, f"out max-abs {d.max():.3e}"
    assert d.mean() <= MEAN_ABS, f"out mean-abs {d.mean():.3e}"
    assert dl.max() <= MAX_ABS, f"lse max-abs {dl.max():.3e}"
    assert dl.mean() <= MEAN_ABS, f"lse mean-abs {dl.mean():.3e}"


def _expected_work(F, T, w, ref, B):
    """Items and (row, key) pairs per head of the two passes, from the block rule: a query block
    of B rows on the padded sequence visits the key blocks that meet its rows' windows, and the
    reference frame's key blocks when some row's window leaves that frame out; every 128-row
    tile of a query block holding a real row is one item."""
    N = F * T
    items = pairs = 0
    r0, r1 = (ref * T // B) * B, -(-((ref + 1) * T) // B) * B
    for q0 in range(0, N, B):
        q1 = min(N, q0 + B)
        fa, fb = q0 // T, (q1 - 1) // T
        lo, hi = max(0, fa - w), min(F - 1, fb + w)
        k0, k1 = (lo * T // B) * B, -(-((hi + 1) * T) // B) * B
        need_ref = not (fb - w <= ref <= fa + w)
        for t0 in range(q0, q1, 128):
            valid = min(128, N - t0)
            items += 1
            pairs += valid * (k1 - k0)
            if need_ref:
                items += 1
                pairs += valid * (r1 - r0)
    return items, pairs


@pytest.mark.parametrize("block", [128, 256])
@pytest.mark.parametrize("name", ["tiny", "small"])
def test_masked_full_parity(dev, oracle_mod, name, block):
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    ref = oracle_mod.attention_full(q, k, v, wl.F, wl.T, wl.w, wl.ref)
    res = _masked(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, block)
    _check(res["out"], res["lse"], ref["out"], ref["lse"])


MASK_EDGE = [
    # H, F, T, D, w, ref, block
    (2, 3, 48, 64, 0, 1, 128),     # frames shorter than a block: a block holds three frames
    (1, 4, 384, 128, 1, 3, 128),   # a frame is three blocks; reference last
    (2, 5, 208, 128, 1, 2, 128),   # block boundaries cut frames; reference in the middle
    (1, 7, 208, 64, 1, 3, 256),    # block 256 and a ragged last block (N = 1456)
    (2, 5, 80, 128, 9, 2, 384),    # window wider than the sequence: no reference pass
    (1, 3, 1200, 128, 1, 0, 512),  # block 512
    (1, 9, 64, 128, 0, 8, 1024),   # largest block: the whole sequence in one padded block
]


@pytest.mark.parametrize("shape", MASK_EDGE)
def test_masked_edge_shapes_full_parity(dev, oracle_mod, shape):
    H, F, T, D, w, ref, block = shape
    q, k, v = make_qkv(H, F * T, D, seed=sum(shape) + 7)
    ref_res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    res = _masked(dev, q, k, v, F, T, w, ref, block, stats=True)
    _check(res["out"], res["lse"], ref_res["out"], ref_res["lse"])
    items, pairs = _expected_work(F, T, w, ref, block)
    assert res["stats"]["items_done"] == H * items
    assert res["stats"]["pairs_visited"] == H * pairs


@pytest.mark.parametrize("name", ["sr28k", "sr57k"])
def test_masked_sampled_parity_full_size(dev, oracle_mod, name):
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    heads, rows = sample_rows(wl, 24)
    ref = oracle_mod.attention_rows(q, k, v, wl.F, wl.T, wl.w, wl.ref, heads, rows)
    res = _masked(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, 128, stats=True)
    _check(res["out"][heads, rows], res["lse"][heads, rows], ref["out"], ref["lse"])
    assert np.isfinite(res["out"]).all() and np.isfinite(res["lse"]).all()
    items, pairs = _expected_work(wl.F, wl.T, wl.w, wl.ref, 128)
    assert res["stats"]["items_done"] == wl.H * items
    assert res["stats"]["pairs_visited"] == wl.H * pairs


def test_masked_agrees_with_frame_aligned(dev):
    # same attention by two layouts: within rounding of each other on every row
    wl = WORKLOADS["small"]
    q, k, v = _inputs("small")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        out_a, lse_a = fsa.forward_ex(qd, kd, vd, plan, "online_max")
        out_m, lse_m = fsa.forward_masked(qd, kd, vd, plan, block=256)
        torch.cuda.synchronize()
    assert float((out_a - out_m).abs().max()) <= MAX_ABS
    assert float((lse_a - lse_m).abs().max()) <= MAX_ABS


def test_masked_repeated_runs_are_bitwise_identical(dev):
    H, F, T, D, w, ref, block = 2, 5, 208, 128, 1, 2, 128
    q, k, v = make_qkv(H, F * T, D, seed=5)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    with fsa.Plan(F, T, w, ref, 16) as plan:
        first = fsa.forward_masked(qd, kd, vd, plan, block=block)
        for _ in range(3):
            again = fsa.forward_masked(qd, kd, vd, plan, block=block)
            torch.cuda.synchronize()
            assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
