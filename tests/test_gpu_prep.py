"""GPU parity of the fused preparation (fsa_prep) against the fp64 CPU oracle.

fsa_prep turns hidden states into the attention's q, k, v (RMS norm, QKV projection, rotary
embedding of q and k, head packing into bf16 [H][N][128]) and produces the norms of the
norm-bound softmax on the way.  Tolerances: q, k, v are bf16, so each element may differ
from the fp64 value by one bf16 step (2^-7 relative) when the fp32 accumulation lands on the
other side of a rounding boundary, plus the fp32 accumulation error of a d_model-term dot
product (below 2e-3 at these sizes).  The norms are compared with fsa_norms run on the
produced q and k (same fp32 arithmetic, other summation order: 2e-6 relative) and with the
oracle's norms of its own rounded q and k (1e-3 relative: a one-step difference in an element
moves a norm by at most |q_i| 2^-7 / ||q||).
"""
import math

import numpy as np
import pytest
import torch

import frame_aligned_block_fsa_b300 as fsa
from frame_aligned_block_fsa_b300.inputs import make_prep_inputs

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from frame_aligned_block_fsa_b300 import build

    build.build()
    fsa.load()
    return torch.device("cuda:0")


def _run_prep(dev, x, w, F, T, w_win, ref, block, H):
    N = F * T
    xd, wd = x.to(dev), w.to(dev)
    qn = torch.full((H, N), -1.0, device=dev)
    km = torch.full((H, F), -1.0, device=dev)
    bd = torch.full((H, N), -1.0, device=dev)
    el = torch.full((H,), 7, dtype=torch.uint8, device=dev)
    st = fsa.new_stats(dev)
    with fsa.Plan(F, T, w_win, ref, block) as plan:
        q, k, v = fsa.prep(xd, wd, plan, H, qnorm=qn, kmax=km, bound=bd, eligible=el, stats=st)
        # fsa_norms on the produced q and k: the norms the separate pass would give
        qn2 = torch.empty_like(qn)
        km2 = torch.empty_like(km)
        bd2 = torch.empty_like(bd)
        el2 = torch.empty_like(el)
        fsa.norms(q, k, plan, qn2, km2, bd2, el2)
        torch.cuda.synchronize()
    stats = fsa.read_stats(st)
    assert stats["error"] == 0, stats
    return {"q": q, "k": k, "v": v, "qnorm": qn, "kmax": km, "bound": bd, "eligible": el,
            "ref_norms": (qn2, km2, bd2, el2)}


def _check_qkv(got, ref):
    g = got.cpu().double().numpy()
    d = np.abs(g - ref)
    tol = 2.0 ** -7 * np.abs(ref) + 2e-3
    assert np.all(d <= tol), f"max excess {(d - tol).max():.3e}"
    assert d.mean() <= 2.0 ** -9 * np.abs(ref).mean()


def _check_norms_consistency(res):
    qn2, km2, bd2, el2 = res["ref_norms"]
    np.testing.assert_allclose(res["qnorm"].cpu().numpy(), qn2.cpu().numpy(), rtol=2e-6)
    np.testing.assert_allclose(res["kmax"].cpu().numpy(), km2.cpu().numpy(), rtol=2e-6)
    np.testing.assert_allclose(res["bound"].cpu().numpy(), bd2.cpu().numpy(), rtol=5e-6)
    assert torch.equal(res["eligible"].cpu(), el2.cpu())


# (F, T, w, ref, block, H, d_model, seed, D): one full row tile; a single ragged tile; three row
# tiles with a ragged last one and frames that do not align with 32-row blocks; T = 16; and
# D = 64 (four heads to a 256-column tile) on ragged shapes
SMALL = [
    (4, 64, 1, 0, 16, 2, 256, 61, 128),
    (3, 80, 1, 2, 80, 4, 192, 62, 128),
    (5, 112, 2, 0, 16, 2, 128, 63, 128),
    (20, 16, 3, 7, 16, 2, 64, 64, 128),
    (5, 112, 2, 0, 16, 4, 128, 69, 64),
    (3, 80, 1, 2, 80, 8, 256, 70, 64),
]


@pytest.mark.parametrize("case", SMALL)
def test_prep_full_parity(dev, oracle_mod, case):
    F, T, w_win, ref, block, H, dm, seed, D = case
    N = F * T
    x, w = make_prep_inputs(N, dm, H, D, seed)
    res = _run_prep(dev, x, w, F, T, w_win, ref, block, H)
    exp = oracle_mod.prep_full(x, w, H, D)
    for name in ("q", "k", "v"):
        _check_qkv(res[name], exp[name])
    _check_norms_consistency(res)
    # the oracle's norms of its own q and k, rounded to bf16 as the kernel stores them
    qr = torch.tensor(exp["q"]).to(torch.bfloat16)
    kr = torch.tensor(exp["k"]).to(torch.bfloat16)
    on = oracle_mod.norms(qr, kr, F, T, w_win, ref)
    np.testing.assert_allclose(res["qnorm"].cpu().double().numpy(), on["qnorm"], rtol=1e-3)
    np.testing.assert_allclose(res["kmax"].cpu().double().numpy(), on["kmax"], rtol=1e-3)
    np.testing.assert_allclose(res["bound"].cpu().double().numpy(), on["bound"], rtol=2e-3)
    worst = on["gap_hat"].max(axis=1)
    margin = np.abs(worst - oracle_mod.DEFAULT_TAU) > 0.05 * oracle_mod.DEFAULT_TAU
    assert np.array_equal(res["eligible"].cpu().numpy()[margin], on["eligible"][margin])


def test_prep_sampled_parity_full_size(dev, oracle_mod):
    # 24 frames x 1200 tokens, 24 heads of 128, d_model 3072 (the 28.8k-token attention's inputs)
    F, T, w_win, ref, block, H, dm = 24, 1200, 2, 0, 80, 24, 3072
    N = F * T
    x, w = make_prep_inputs(N, dm, H, D, seed=65)
    res = _run_prep(dev, x, w, F, T, w_win, ref, block, H)
    g = torch.Generator().manual_seed(66)
    special = [0, 1, 31, 32, 255, 256, 1199, 1200, 1201, 14399, 14400, 28543, 28544, 28799]
    rows = np.array(special + torch.randint(0, N, (18,), generator=g).tolist(), dtype=np.int64)
    exp = oracle_mod.prep_rows(x, w, H, D, rows)
    for name in ("q", "k", "v"):
        got = res[name][:, torch.as_tensor(rows, device=res[name].device)].transpose(0, 1)  # [R][H][D]
        _check_qkv(got, exp[name])
    _check_norms_consistency(res)


def test_prep_is_deterministic_and_feeds_the_attention(dev):
    F, T, w_win, ref, block, H, dm = 6, 400, 1, 0, 80, 4, 512
    N = F * T
    x, w = make_prep_inputs(N, dm, H, D, seed=67)
    a = _run_prep(dev, x, w, F, T, w_win, ref, block, H)
    b = _run_prep(dev, x, w, F, T, w_win, ref, block, H)
    for name in ("q", "k", "v", "qnorm", "kmax", "bound", "eligible"):
        assert torch.equal(a[name], b[name]), name
    # The attention with the prep's norms matches the attention with fsa_norms' norms.  The two
    # bounds differ in the last bits (summation order), which moves exp(s - bound) by a relative
    # 1e-6 and flips the bf16 rounding of a few P values: out moves by far less than one bf16
    # step of P (2^-8), the lse (fp32 row sum) by rounding only.
    with fsa.Plan(F, T, w_win, ref, block) as plan:
        o1, l1 = fsa.forward_ex(a["q"], a["k"], a["v"], plan, "norm_bound", bound=a["bound"], eligible=a["eligible"])
        o2, l2 = fsa.forward(a["q"], a["k"], a["v"], plan, "norm_bound")
        torch.cuda.synchronize()
    do = (o1 - o2).abs()
    assert float(do.max()) <= 1e-3 and float(do.mean()) <= 1e-5
    assert float((l1 - l2).abs().max()) <= 1e-4


@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
def test_prep_then_attention_matches_the_oracle_chain(dev, oracle_mod, mode):
    # The whole widened path: hidden states -> fsa_prep (q, k, v, bound, eligibility) ->
    # attention with those norms, against the oracle's prep (rounded to bf16, as stored) followed
    # by the oracle's attention.  A q, k or v element may sit one bf16 step from the oracle's
    # rounding; that moves out and lse far less than the attention tolerance.
    F, T, w_win, ref, block, H, dm = 4, 96, 1, 2, 32, 2, 256
    N = F * T
    x, w = make_prep_inputs(N, dm, H, D, seed=68)
    exp = oracle_mod.prep_full(x, w, H, D)
    qr, kr, vr = (torch.tensor(exp[n]).to(torch.bfloat16) for n in ("q", "k", "v"))
    att = oracle_mod.attention_full(qr, kr, vr, F, T, w_win, ref)
    with fsa.Plan(F, T, w_win, ref, block) as plan:
        bd = torch.empty((H, N), device=dev)
        el = torch.empty(H, dtype=torch.uint8, device=dev)
        q, k, v = fsa.prep(x.to(dev), w.to(dev), plan, H, bound=bd, eligible=el)
        st = fsa.new_stats(dev)
        out, lse = fsa.forward_ex(q, k, v, plan, mode, bound=bd, eligible=el, stats=st)
        torch.cuda.synchronize()
    stats = fsa.read_stats(st)
    assert stats["error"] == 0 and stats["fallback_heads"] == 0
    d = np.abs(out.cpu().double().numpy() - att["out"])
    dl = np.abs(lse.cpu().double().numpy() - att["lse"])
    assert d.max() <= 1e-2 and d.mean() <= 1e-3, (d.max(), d.mean())
    assert dl.max() <= 1e-2 and dl.mean() <= 1e-3, (dl.max(), dl.mean())
