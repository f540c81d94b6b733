"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: hand-derived
golden fixtures, brute force written independently in Python, closed forms,
library routines (numpy / scipy) and invariants of softmax attention.
"""
import math
import os

import numpy as np
import pytest
import torch

from frame_aligned_block_fsa_b300.inputs import make_qkv
from frame_aligned_block_fsa_b300.workloads import WORKLOADS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


# --------------------------------------------------------------------------- plan
@pytest.mark.parametrize("name", sorted(f for f in os.listdir(GOLDEN) if f.startswith("plan_")))
def test_plan_matches_hand_derived_golden(oracle_mod, name):
    g = _read_golden(name)
    F, T, w, ref, B = (int(g[k][0]) for k in ("F", "T", "w", "ref", "block"))
    row_ptr, col_idx = oracle_mod.plan(F, T, w, ref, B)
    assert row_ptr.tolist() == [int(x) for x in g["row_ptr"]]
    assert col_idx.tolist() == [int(x) for x in g["col_idx"]]


# Hand-counted frame pairs (sum over query frames of |S(f)|) for the five workloads:
#   tiny   F=8,  w=1: 2+3+4*5+3                      = 28
#   small  F=16, w=2: 3+4+5 + 6*11 + 5+4             = 87
#   sr28k  F=24, w=2: 3+4+5 + 6*19 + 5+4             = 135
#   sr57k  F=16, w=1: 2+3 + 4*13 + 3                 = 60
#   stress F=24, w=4: 5+6+7+8+9 + 10*15 + 9+8+7+6    = 215
HAND_PAIRS = {"tiny": 28, "small": 87, "sr28k": 135, "sr57k": 60, "stress": 215}


@pytest.mark.parametrize("name", list(HAND_PAIRS))
def test_frame_pairs_and_nnz_closed_form(oracle_mod, name):
    wl = WORKLOADS[name]
    assert oracle_mod.active_frame_pairs(wl.F, wl.w, wl.ref) == HAND_PAIRS[name]
    row_ptr, col_idx = oracle_mod.plan(wl.F, wl.T, wl.w, wl.ref, wl.block)
    per_frame = wl.T // wl.block
    assert len(col_idx) == HAND_PAIRS[name] * per_frame * per_frame
    assert row_ptr[-1] == len(col_idx)
    # within every row the key blocks ascend strictly
    for r in range(len(row_ptr) - 1):
        seg = col_idx[row_ptr[r]:row_ptr[r + 1]]
        assert np.all(np.diff(seg) > 0)


def test_plan_rejects_partial_blocks(oracle_mod):
    # T=24 with block 16: blocks straddle frame boundaries -> partial blocks exist.
    with pytest.raises(ValueError):
        oracle_mod.plan(4, 24, 1, 0, 16)


def test_plan_brute_force_small(oracle_mod):
    # independent restatement: a block pair is active iff its first token pair is allowed
    for (F, T, w, ref, B) in [(6, 32, 1, 3, 16), (7, 48, 2, 6, 16), (5, 96, 0, 0, 48), (9, 16, 3, 4, 16)]:
        row_ptr, col_idx = oracle_mod.plan(F, T, w, ref, B)
        nb = F * T // B
        expect_ptr, expect_idx = [0], []
        for qb in range(nb):
            fq = qb * B // T
            for kb in range(nb):
                fk = kb * B // T
                if abs(fq - fk) <= w or fk == ref:
                    expect_idx.append(kb)
            expect_ptr.append(len(expect_idx))
        assert row_ptr.tolist() == expect_ptr
        assert col_idx.tolist() == expect_idx


# ---------------------------------------------------------------------- attention
def test_attention_matches_hand_worked_example(oracle_mod):
    g = _read_golden("attention_F2_T1_D1.txt")
    q = _bf16(g["q"]).reshape(1, 2, 1)
    k = _bf16(g["k"]).reshape(1, 2, 1)
    v = _bf16(g["v"]).reshape(1, 2, 1)
    res = oracle_mod.attention_full(q, k, v, F=2, T=1, w=0, ref=0, scale=1.0)
    np.testing.assert_allclose(res["out"][0, :, 0], g["out"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(res["lse"][0], g["lse"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(res["bound"][0], g["bound"], rtol=0, atol=1e-14)


def _brute_force(q, k, v, F, T, w, ref, scale):
    """Pure-Python restatement: enumerate allowed (i, j) from the frame rule directly."""
    H, N, D = q.shape
    out = np.zeros((H, N, D))
    lse = np.zeros((H, N))
    for h in range(H):
        for i in range(N):
            fi = i // T
            keys = [j for j in range(N) if abs(fi - j // T) <= w or j // T == ref]
            logits = [scale * sum(q[h, i, d] * k[h, j, d] for d in range(D)) for j in keys]
            m = max(logits)
            e = [math.exp(s - m) for s in logits]
            l = math.fsum(e)
            for d in range(D):
                out[h, i, d] = math.fsum(e[t] * v[h, j, d] for t, j in enumerate(keys)) / l
            lse[h, i] = m + math.log(l)
    return out, lse


@pytest.mark.parametrize("case", [
    (2, 3, 4, 1, 8, 1, 0), (1, 4, 3, 0, 4, 1, 2), (2, 3, 5, 2, 8, 7, 1), (1, 2, 8, 0, 16, 0, 1),
])
def test_attention_matches_brute_force_tiny(oracle_mod, case):
    H, F, T, w, D, seed, ref = case
    q, k, v = make_qkv(H, F * T, D, seed)
    ref_out, ref_lse = _brute_force(_f64(q), _f64(k), _f64(v), F, T, w, ref, 1 / math.sqrt(D))
    res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    np.testing.assert_allclose(res["out"], ref_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["lse"], ref_lse, rtol=1e-12, atol=1e-13)


def test_dense_window_is_textbook_attention(oracle_mod):
    from scipy.special import logsumexp, softmax

    H, F, T, D = 2, 4, 16, 16
    q, k, v = make_qkv(H, F * T, D, seed=5)
    for w in (F - 1, F + 3):
        res = oracle_mod.attention_full(q, k, v, F, T, w, ref=1)
        qq, kk, vv = _f64(q), _f64(k), _f64(v)
        logits = np.einsum("hnd,hmd->hnm", qq, kk) / math.sqrt(D)
        expect = np.einsum("hnm,hmd->hnd", softmax(logits, axis=-1), vv)
        np.testing.assert_allclose(res["out"], expect, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(res["lse"], logsumexp(logits, axis=-1), rtol=1e-12, atol=1e-12)



def test_attention_is_invariant_to_key_order_within_frames(oracle_mod):
    # Permuting the tokens of every frame (the same permutation for k and v) leaves each
    # frame's key set, and so every softmax, unchanged.
    H, F, T, D, w, ref = 2, 5, 16, 32, 1, 3
    q, k, v = make_qkv(H, F * T, D, seed=12)
    g = torch.Generator().manual_seed(13)
    perm = torch.cat([f * T + torch.randperm(T, generator=g) for f in range(F)])
    a = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    b = oracle_mod.attention_full(q, k[:, perm].contiguous(), v[:, perm].contiguous(), F, T, w, ref)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-13, atol=1e-13)


def test_key_translation_moves_lse_only(oracle_mod):
    # Adding one vector m to every key adds c <q_i, m> to every logit of row i: the softmax and
    # out do not change, and lse moves by exactly that row constant.  Integer-valued keys keep
    # the shifted keys exact in bf16.
    H, F, T, D, w, ref = 2, 4, 16, 16, 1, 0
    q, _, v = make_qkv(H, F * T, D, seed=14)
    rng = np.random.default_rng(15)
    z = rng.integers(-3, 4, size=(H, F * T, D)).astype(np.float32)
    m = rng.integers(-8, 9, size=(H, 1, D)).astype(np.float32)
    k0 = torch.tensor(z).to(torch.bfloat16)
    k1 = torch.tensor(z + m).to(torch.bfloat16)
    assert torch.equal(k1.float(), torch.tensor(z + m))
    a = oracle_mod.attention_full(q, k0, v, F, T, w, ref)
    b = oracle_mod.attention_full(q, k1, v, F, T, w, ref)
    shift = np.einsum("hnd,hd->hn", _f64(q), m[:, 0, :].astype(np.float64)) / math.sqrt(D)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b["lse"] - a["lse"], shift, rtol=1e-10, atol=1e-10)

def _allowed_count(F, T, w, ref, f):
    return T * sum(1 for g in range(F) if abs(f - g) <= w or g == ref)


def test_zero_query_gives_mean_of_attended_values(oracle_mod):
    H, F, T, D, w, ref = 1, 5, 8, 16, 1, 3
    _, k, v = make_qkv(H, F * T, D, seed=7)
    q = torch.zeros_like(k)
    res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    vv = _f64(v)[0]
    for i in range(F * T):
        f = i // T
        sel = [j for j in range(F * T) if abs(f - j // T) <= w or j // T == ref]
        np.testing.assert_allclose(res["out"][0, i], vv[sel].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert res["lse"][0, i] == pytest.approx(math.log(_allowed_count(F, T, w, ref, f)), abs=1e-13)


def test_constant_values_give_constant_output(oracle_mod):
    H, F, T, D = 2, 4, 8, 16
    q, k, _ = make_qkv(H, F * T, D, seed=8)
    v = torch.full((H, F * T, D), -1.75, dtype=torch.bfloat16)
    res = oracle_mod.attention_full(q, k, v, F, T, 1, 0)
    np.testing.assert_allclose(res["out"], -1.75, rtol=0, atol=1e-14)


def test_identical_keys_give_uniform_weights(oracle_mod):
    H, F, T, D, w, ref = 1, 6, 4, 8, 1, 5
    q, _, v = make_qkv(H, F * T, D, seed=9)
    krow = make_qkv(1, 1, D, seed=10)[1][0, 0]
    k = krow.expand(H, F * T, D).contiguous()
    res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    qq, kk, vv = _f64(q)[0], _f64(k)[0], _f64(v)[0]
    for i in range(F * T):
        f = i // T
        sel = [j for j in range(F * T) if abs(f - j // T) <= w or j // T == ref]
        s = float(qq[i] @ kk[0]) / math.sqrt(D)
        np.testing.assert_allclose(res["out"][0, i], vv[sel].mean(axis=0), rtol=1e-12, atol=1e-13)
        assert res["lse"][0, i] == pytest.approx(s + math.log(len(sel)), rel=1e-13, abs=1e-13)


def test_weights_sum_to_one_and_vanish_off_mask(oracle_mod):
    # V rows are the basis vectors e_j, so out_i is the weight row p_i itself.
    F, T, w, ref = 4, 3, 1, 3
    N = F * T
    D = 16
    q, k, _ = make_qkv(1, N, D, seed=11)
    v = torch.zeros((1, N, D), dtype=torch.bfloat16)
    for j in range(N):
        v[0, j, j] = 1.0
    res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    p = res["out"][0]
    for i in range(N):
        assert math.fsum(p[i]) == pytest.approx(1.0, abs=1e-12)
        for j in range(N):
            allowed = abs(i // T - j // T) <= w or j // T == ref
            if allowed:
                assert p[i, j] > 0.0
            else:
                assert p[i, j] == 0.0
        assert np.all(p[i, N:] == 0.0)


@pytest.mark.parametrize("kind", ["normal", "stress"])
def test_bound_form_equals_max_form_and_dominates(oracle_mod, kind):
    H, F, T, D, w, ref = 2, 6, 16, 32, 1, 0
    q, k, v = make_qkv(H, F * T, D, seed=13, kind=kind)
    res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    ok = ~res["underflow"]
    assert ok.any()
    # Cauchy-Schwarz: the row's own bound is never below its true max
    assert np.all(res["bound"] >= res["rowmax"] - 1e-12 * np.abs(res["bound"]))
    # exact-arithmetic equality of the two softmax forms on rows that do not underflow
    np.testing.assert_allclose(res["out_bound"][ok], res["out"][ok], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(res["lse_bound"][ok], res["lse"][ok], rtol=1e-12, atol=1e-12)


def test_bound_is_tight_for_parallel_key(oracle_mod):
    # a key equal to the query and of the largest norm attains the bound exactly
    D = 4
    q = _bf16([[1, 2, -2, 4], [0.5, 0.5, 0.5, 0.5]]).reshape(1, 2, D)
    k = _bf16([[1, 2, -2, 4], [0, 1, 0, 1]]).reshape(1, 2, D)
    v = _bf16([[1, 0, 0, 0], [0, 1, 0, 0]]).reshape(1, 2, D)
    res = oracle_mod.attention_full(q, k, v, F=1, T=2, w=0, ref=0)
    assert res["gap"][0, 0] == pytest.approx(0.0, abs=1e-12)
    assert res["bound"][0, 0] == pytest.approx(25.0 / 2.0, abs=1e-12)  # |q|^2 / sqrt(4)


def test_underflow_flag_and_nan_bound_form(oracle_mod):
    # D=1, scale 1, T=1 (one token per frame), w=0, reference frame 1.
    #   frame 0 -> keys {0, 1}: s = -81, -36; m = -36; bound = 9*9 = 81;  gap = 117
    #   frame 1 -> keys {1}:    s = -36;      m = -36; bound = 9*4 = 36;  gap = 72
    #   frame 2 -> keys {1, 2}: s = -36, 18;  m = 18;  bound = 9*4 = 36;  gap = 18
    #   frame 3 -> keys {1, 3}: s = -120, -900; m = -120; bound = 900;  gap = 1020
    # fp32 underflow iff gap >= 126 ln 2 = 87.34; fp64 itself underflows only past ~745,
    # where the bound form of the oracle turns into 0/0.
    q = _bf16([9, 9, 9, 30]).reshape(1, 4, 1)
    k = _bf16([-9, -4, 2, -30]).reshape(1, 4, 1)
    v = _bf16([1, 2, 3, 4]).reshape(1, 4, 1)
    res = oracle_mod.attention_full(q, k, v, F=4, T=1, w=0, ref=1, scale=1.0)
    np.testing.assert_allclose(res["gap"][0], [117.0, 72.0, 18.0, 1020.0], atol=1e-12)
    assert res["underflow"][0].tolist() == [True, False, False, True]
    assert res["out"][0, 0, 0] == pytest.approx(2.0, abs=1e-12)
    assert res["out_bound"][0, 0, 0] == pytest.approx(2.0, abs=1e-12)
    assert res["out"][0, 3, 0] == pytest.approx(2.0, abs=1e-12)
    assert math.isnan(res["out_bound"][0, 3, 0])
    assert res["out"][0, 2, 0] == pytest.approx((3 + 2 * math.exp(-54)) / (1 + math.exp(-54)), abs=1e-14)


# -------------------------------------------------------------------------- norms
@pytest.mark.parametrize("kind", ["normal", "stress"])
def test_norms_against_library_routines_and_gap_bound(oracle_mod, kind):
    H, F, T, D, w, ref = 2, 5, 16, 32, 1, 2
    q, k, v = make_qkv(H, F * T, D, seed=21, kind=kind)
    nm = oracle_mod.norms(q, k, F, T, w, ref)
    qq, kk = _f64(q), _f64(k)
    np.testing.assert_allclose(nm["qnorm"], np.linalg.norm(qq, axis=-1), rtol=1e-14)
    kn = np.linalg.norm(kk, axis=-1).reshape(H, F, T)
    np.testing.assert_allclose(nm["kmax"], kn.max(axis=-1), rtol=1e-14)
    att = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    # the per-frame-max route and the per-row-key-set route give the same bound
    np.testing.assert_allclose(nm["bound"], att["bound"], rtol=1e-13)
    # the eligibility statistic bounds the true gap from above
    assert np.all(nm["gap_hat"] >= att["gap"] - 1e-9)
    # eligibility is the threshold test on the per-head worst gap bound
    for tau in (0.5, 5.0, 50.0, 1e6):
        e = oracle_mod.norms(q, k, F, T, w, ref, tau=tau)["eligible"]
        assert e.tolist() == [int(x <= tau) for x in nm["gap_hat"].max(axis=1)]


def test_centred_norms_hand_derived(oracle_mod):
    # D=1, T=1, scale 1, w=0, reference frame 0.  Keys 1, 2, 6: head mean mu = 3, centred
    # key norms |k - mu| = 2, 1, 3.  Queries 1, -1, 2.
    #   frame 0: S = {0}     Kc = 2  bound = 1*2 + 1*3 = 5      kbar = 1    gap_hat = 5 - 1 = 4
    #   frame 1: S = {0, 1}  Kc = 2  bound = 1*2 + (-1)*3 = -1  kbar = 1.5  gap_hat = -1 + 1.5 = 0.5
    #   frame 2: S = {0, 2}  Kc = 3  bound = 2*3 + 2*3 = 12     kbar = 3.5  gap_hat = 12 - 7 = 5
    # Row maxima: 1, -1, 12 (frames 1 and 2 meet their centred bound exactly).  Without
    # centring the bounds are 1*1, 1*2, 2*6, the key maxima 1, 2, 6 and the gap statistics
    # 1 - 1, 2 + 1.5, 12 - 7.
    q = _bf16([1, -1, 2]).reshape(1, 3, 1)
    k = _bf16([1, 2, 6]).reshape(1, 3, 1)
    c = oracle_mod.norms(q, k, F=3, T=1, w=0, ref=0, scale=1.0, tau=4.5, center=True)
    np.testing.assert_allclose(c["kmax"][0], [2.0, 1.0, 3.0], atol=1e-15)
    np.testing.assert_allclose(c["bound"][0], [5.0, -1.0, 12.0], atol=1e-15)
    np.testing.assert_allclose(c["gap_hat"][0], [4.0, 0.5, 5.0], atol=1e-15)
    assert c["eligible"].tolist() == [0]
    u = oracle_mod.norms(q, k, F=3, T=1, w=0, ref=0, scale=1.0, center=False)
    np.testing.assert_allclose(u["kmax"][0], [1.0, 2.0, 6.0], atol=1e-15)
    np.testing.assert_allclose(u["bound"][0], [1.0, 2.0, 12.0], atol=1e-15)
    # uncentred gap statistic bound - q kbar_S: 1 - 1*1, 2 - (-1)*1.5, 12 - 2*3.5
    np.testing.assert_allclose(u["gap_hat"][0], [0.0, 3.5, 5.0], atol=1e-15)
    # eligible iff the worst gap statistic <= tau, the boundary included (5 is exact here)
    for tau, elig in ((4.9, 0), (5.0, 1), (5.1, 1)):
        assert oracle_mod.norms(q, k, F=3, T=1, w=0, ref=0, scale=1.0, tau=tau)["eligible"].tolist() == [elig]
    att = oracle_mod.attention_full(q, k, k, F=3, T=1, w=0, ref=0, scale=1.0)
    np.testing.assert_allclose(att["rowmax"][0], [1.0, -1.0, 12.0], atol=1e-15)


def _integer_keys(H, N, D, seed, offset):
    # small integers: every sum below is exact in bf16 and fp64
    g = np.random.default_rng(seed)
    z = g.integers(-4, 5, size=(H, N, D)).astype(np.float32)
    m = g.integers(-offset, offset + 1, size=(H, 1, D)).astype(np.float32)
    return z, m


def test_centred_bound_is_translation_invariant(oracle_mod):
    # Shifting every key of a head by one vector m moves each centred bound by exactly
    # c <q, m> and leaves the centred key norms and the gap bound unchanged; the uncentred
    # bound has no such property.  The centred bound still bounds the brute-force row max.
    H, F, T, D, w, ref = 2, 6, 16, 32, 1, 3
    z, m = _integer_keys(H, F * T, D, seed=5, offset=40)
    q, _, v = make_qkv(H, F * T, D, seed=22)
    k0, k1 = _bf16(z), _bf16(z + m)
    assert torch.equal(k1.float(), torch.tensor(z + m))  # the shifted keys are exact
    n0 = oracle_mod.norms(q, k0, F, T, w, ref, center=True)
    n1 = oracle_mod.norms(q, k1, F, T, w, ref, center=True)
    c = 1.0 / math.sqrt(D)
    qm = np.einsum("hnd,hd->hn", _f64(q), m[:, 0, :].astype(np.float64))
    np.testing.assert_allclose(n1["kmax"], n0["kmax"], rtol=1e-12)
    np.testing.assert_allclose(n1["bound"] - n0["bound"], c * qm, atol=1e-9)
    np.testing.assert_allclose(n1["gap_hat"], n0["gap_hat"], atol=1e-9)
    att = oracle_mod.attention_full(q, k1, v, F, T, w, ref)
    assert np.all(n1["bound"] >= att["rowmax"] - 1e-9)
    assert np.all(n1["gap_hat"] >= n1["bound"] - att["rowmax"] - 1e-9)
    # the common component inflates the uncentred gap bound, not the centred one
    u1 = oracle_mod.norms(q, k1, F, T, w, ref, center=False)
    assert n1["gap_hat"].max() < 0.5 * u1["gap_hat"].max()


def test_centred_equals_uncentred_for_zero_mean_keys(oracle_mod):
    # keys in +-pairs: the head mean is exactly zero, so centring changes nothing
    H, F, T, D, w, ref = 2, 4, 16, 64, 1, 0
    q, k, _ = make_qkv(H, F * T, D, seed=23)
    kk = k.clone()
    kk[:, 1::2, :] = -k[:, 0::2, :]
    a = oracle_mod.norms(q, kk, F, T, w, ref, tau=10.0, center=True)
    b = oracle_mod.norms(q, kk, F, T, w, ref, tau=10.0, center=False)
    for name in ("qnorm", "kmax", "gap_hat", "eligible"):
        np.testing.assert_array_equal(a[name], b[name])
    np.testing.assert_allclose(a["bound"], b["bound"], rtol=1e-15)
    for tau in (0.5, 5.0, 50.0):
        e = oracle_mod.norms(q, kk, F, T, w, ref, tau=tau, center=True)["eligible"]
        assert e.tolist() == [int(x <= tau) for x in a["gap_hat"].max(axis=1)]

# --------------------------------------------------------------------------- prep
def test_prep_hand_derived_rotation(oracle_mod):
    # H = 1, D = 4, d_model = 4, eps = 0, base 100: theta = (1, 1/10).  W = [I; 2I; 3I] (q, k,
    # v).  Token 1 is x = (2, 0, 0, 2): rms = sqrt(8/4) = sqrt 2, xhat = (sqrt2, 0, 0, sqrt2).
    # Pairs (0, 2) and (1, 3) turn by 1 and 0.1 rad at position 1:
    #   q = (s cos1 - 0 sin1, 0 cos.1 - s sin.1, s sin1 + 0 cos1, 0 sin.1 + s cos.1), s = sqrt2
    # k is 2 q, v = 3 xhat unrotated; token 0 (position 0) is not rotated at all.
    x = _bf16([[1, -1, 1, -1], [2, 0, 0, 2]])
    eye = np.eye(4, dtype=np.float32)
    w = _bf16(np.concatenate([eye, 2 * eye, 3 * eye]))
    r = oracle_mod.prep_full(x, w, H=1, D=4, eps=0.0, base=100.0)
    s = math.sqrt(2.0)
    q1 = [s * math.cos(1.0), -s * math.sin(0.1), s * math.sin(1.0), s * math.cos(0.1)]
    np.testing.assert_allclose(r["q"][0, 1], q1, atol=1e-15)
    np.testing.assert_allclose(r["k"][0, 1], 2 * np.asarray(q1), atol=1e-15)
    np.testing.assert_allclose(r["v"][0, 1], [3 * s, 0, 0, 3 * s], atol=1e-15)
    np.testing.assert_allclose(r["q"][0, 0], [1, -1, 1, -1], atol=1e-15)  # rms 1, no rotation
    np.testing.assert_allclose(r["v"][0, 0], [3, -3, 3, -3], atol=1e-15)
    # eps enters under the root: with eps = 1 token 1 has rms sqrt(8/4 + 1) = sqrt 3
    r1 = oracle_mod.prep_full(x, w, H=1, D=4, eps=1.0, base=100.0)
    np.testing.assert_allclose(r1["v"][0, 1], [6 / math.sqrt(3), 0, 0, 6 / math.sqrt(3)], atol=1e-15)
    np.testing.assert_allclose(r1["v"][0, 0], [3 / math.sqrt(2), -3 / math.sqrt(2), 3 / math.sqrt(2),
                                               -3 / math.sqrt(2)], atol=1e-15)


def _numpy_projection(x, w, eps):
    xx = _f64(x)
    xh = xx / np.sqrt((xx * xx).mean(axis=1, keepdims=True) + eps)
    return xh @ _f64(w).T  # [N][3 H D]


def test_prep_projection_norms_and_relative_positions(oracle_mod):
    from frame_aligned_block_fsa_b300.inputs import make_prep_inputs

    N, dm, H, D = 40, 96, 2, 16
    x, w = make_prep_inputs(N, dm, H, D, seed=51)
    # tokens 30..39 repeat tokens 0..9 ten positions later
    x[30:40] = x[0:10]
    r = oracle_mod.prep_full(x, w, H, D)
    y = _numpy_projection(x, w, oracle_mod.PREP_EPS).reshape(N, 3, H, D).transpose(1, 2, 0, 3)
    # v and every row at position 0 are the plain projection (numpy matmul)
    np.testing.assert_allclose(r["v"], y[2], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["q"][:, 0], y[0][:, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["k"][:, 0], y[1][:, 0], rtol=1e-12, atol=1e-12)
    # the rotation keeps every head row's norm
    np.testing.assert_allclose(np.linalg.norm(r["q"], axis=-1), np.linalg.norm(y[0], axis=-1), rtol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(r["k"], axis=-1), np.linalg.norm(y[1], axis=-1), rtol=1e-12)
    # logits depend on the positions only through their difference
    a = np.einsum("hmd,hnd->hmn", r["q"][:, 0:10], r["k"][:, 0:10])
    b = np.einsum("hmd,hnd->hmn", r["q"][:, 30:40], r["k"][:, 30:40])
    np.testing.assert_allclose(b, a, rtol=1e-9, atol=1e-9)
    # ... and do change with it (the rotation is not the identity)
    assert np.abs(r["q"][:, 30] - r["q"][:, 0]).max() > 1e-2


def test_prep_rms_norm_scale_invariance_and_row_sampling(oracle_mod):
    from frame_aligned_block_fsa_b300.inputs import make_prep_inputs

    N, dm, H, D = 24, 64, 2, 8
    x, w = make_prep_inputs(N, dm, H, D, seed=52)
    a = oracle_mod.prep_full(x, w, H, D, eps=0.0)
    b = oracle_mod.prep_full((x.float() * 4).to(torch.bfloat16), w, H, D, eps=0.0)  # exact in bf16
    for name in ("q", "k", "v"):
        np.testing.assert_allclose(b[name], a[name], rtol=1e-13, atol=1e-13)
    rows = np.array([23, 0, 7, 7], dtype=np.int64)
    s = oracle_mod.prep_rows(x, w, H, D, rows, eps=0.0)
    for name in ("q", "k", "v"):
        np.testing.assert_array_equal(s[name], a[name][:, rows].transpose(1, 0, 2))

def test_active_flops_formula_matches_enumeration(oracle_mod):
    wl = WORKLOADS["small"]
    row_ptr, col_idx = oracle_mod.plan(wl.F, wl.T, wl.w, wl.ref, wl.block)
    # every active block pair contributes QK^T and PV: 2 * (2 * B * B * D) flops per head
    expect = len(col_idx) * 4 * wl.block * wl.block * wl.D * wl.H
    assert oracle_mod.active_flops(wl.F, wl.T, wl.w, wl.ref, wl.H, wl.D) == expect
