"""GPU parity: the CUDA path, called through the C ABI, against the fp64 CPU oracle.

Tolerances.  For unit-variance inputs the fp32 outputs must lie within max-abs 1e-2 and
mean-abs 1e-3 of the oracle (out and lse).  For the stress inputs (log-normal row norms,
8x outlier keys) logits reach ~1e4, and fp32 accumulation of a D-term dot product carries
an error of order sqrt(D) * 2^-24 * c ||q|| ||k|| <= sqrt(D) * 2^-24 * bound_i; the stress
tolerance adds that term (times a safety factor 8, and times max|v| for out).
"""
import math

import numpy as np
import pytest
import torch

import frame_aligned_block_fsa_b300 as fsa
from frame_aligned_block_fsa_b300.inputs import make_qkv, make_workload_inputs, sample_rows
from frame_aligned_block_fsa_b300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
U32 = 2.0 ** -24
UNDERFLOW_GAP = 126.0 * math.log(2.0)

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


def _oracle_full(oracle_mod, name):
    key = ("full", name)
    if key not in _cache:
        wl = WORKLOADS[name]
        q, k, v = _inputs(name)
        _cache[key] = oracle_mod.attention_full(q, k, v, wl.F, wl.T, wl.w, wl.ref)
    return _cache[key]


def _oracle_sampled(oracle_mod, name, per_head):
    key = ("rows", name, per_head)
    if key not in _cache:
        wl = WORKLOADS[name]
        q, k, v = _inputs(name)
        heads, rows = sample_rows(wl, per_head)
        _cache[key] = (heads, rows, oracle_mod.attention_rows(q, k, v, wl.F, wl.T, wl.w, wl.ref, heads, rows))
    return _cache[key]


def _gpu(dev, q, k, v, F, T, w, ref, block, mode, key_tile=0, tau=None, rowmax=False, stats=False,
         center_keys=False):
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    H, N, D = q.shape
    with fsa.Plan(F, T, w, ref, block) as plan:
        if key_tile:
            plan.set_key_tile(key_tile)
        if center_keys:
            plan.set_center_keys(True)
        if tau is not None:
            plan.set_tau(tau)
        rm = torch.full((H, N), float("nan"), device=dev) if rowmax else None
        st = fsa.new_stats(dev) if stats else None
        out, lse = fsa.forward_ex(qd, kd, vd, plan, mode, rowmax=rm, stats=st)
        torch.cuda.synchronize()
    res = {"out": out.cpu().double().numpy(), "lse": lse.cpu().double().numpy(), "out_t": out, "lse_t": lse}
    if rowmax:
        res["rowmax"] = rm.cpu().double().numpy()
    if stats:
        res["stats"] = fsa.read_stats(st)
        assert res["stats"]["error"] == 0, res["stats"]
    return res


def _check(out, lse, ref_out, ref_lse, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    d = np.abs(out - ref_out)
    dl = np.abs(lse - ref_lse)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert d.max() <= max_abs, f"out max-abs {d.max():.3e}"
    assert d.mean() <= mean_abs, f"out mean-abs {d.mean():.3e}"
    assert dl.max() <= max_abs, f"lse max-abs {dl.max():.3e}"
    assert dl.mean() <= mean_abs, f"lse mean-abs {dl.mean():.3e}"


# --------------------------------------------------------------------------- boundary
def test_bounded_wait_gives_up_with_timeout_status(dev):
    assert fsa.selftest_wait_timeout(200_000) == fsa.FSA_ERR_TIMEOUT
    # the context stays usable afterwards
    x = torch.ones(1024, device=dev)
    assert float(x.sum()) == 1024.0


def test_prep_grid_barrier_opens_and_times_out(dev):
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for ctas in (2, sms):
        # every CTA arrives: the barrier opens, nothing is reported
        r = fsa.selftest_grid_timeout(50_000_000, ctas, 0)
        assert r == {"status": 0, "site": 0, "gave_up": 0, "arrived": ctas}, r
        # one arrival never comes: every CTA gives up with the grid-barrier site
        r = fsa.selftest_grid_timeout(200_000, ctas, 1)
        assert r == {"status": fsa.FSA_ERR_TIMEOUT, "site": 16, "gave_up": ctas, "arrived": ctas}, r
    # the context stays usable afterwards
    x = torch.ones(1024, device=dev)
    assert float(x.sum()) == 1024.0


# ----------------------------------------------------------------------- full parity
@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
@pytest.mark.parametrize("name", ["tiny", "small"])
def test_forward_full_parity(dev, oracle_mod, name, mode):
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    ref = _oracle_full(oracle_mod, name)
    res = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, mode, stats=True)
    _check(res["out"], res["lse"], ref["out"], ref["lse"])
    assert res["stats"]["fallback_heads"] == 0


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_norms_parity(dev, oracle_mod, name):
    wl = WORKLOADS[name]
    q, k, _ = _inputs(name)
    H, N, D = q.shape
    on = oracle_mod.norms(q, k, wl.F, wl.T, wl.w, wl.ref)
    qd, kd = q.to(dev), k.to(dev)
    qn = torch.empty((H, N), device=dev)
    km = torch.empty((H, wl.F), device=dev)
    bd = torch.empty((H, N), device=dev)
    el = torch.empty(H, dtype=torch.uint8, device=dev)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        fsa.norms(qd, kd, plan, qn, km, bd, el)
        torch.cuda.synchronize()
    np.testing.assert_allclose(qn.cpu().double().numpy(), on["qnorm"], rtol=2e-6)
    np.testing.assert_allclose(km.cpu().double().numpy(), on["kmax"], rtol=2e-6)
    np.testing.assert_allclose(bd.cpu().double().numpy(), on["bound"], rtol=5e-6)
    worst = on["gap_hat"].max(axis=1)
    margin = np.abs(worst - oracle_mod.DEFAULT_TAU) > 1e-3 * oracle_mod.DEFAULT_TAU
    assert np.array_equal(el.cpu().numpy()[margin], on["eligible"][margin])


# -------------------------------------------------------------------- sampled parity
@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
@pytest.mark.parametrize("name", ["sr28k", "sr57k"])
def test_forward_sampled_parity_full_size(dev, oracle_mod, name, mode):
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    heads, rows, ref = _oracle_sampled(oracle_mod, name, per_head=24)
    res = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, mode, stats=True)
    _check(res["out"][heads, rows], res["lse"][heads, rows], ref["out"], ref["lse"])
    assert res["stats"]["underflow_rows"] == 0
    # properties that hold at every row: finite, lse at least the mean logit bound
    assert np.isfinite(res["out"]).all() and np.isfinite(res["lse"]).all()


def test_stress_fallback_and_underflow(dev, oracle_mod):
    name = "stress"
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    H, N, D = q.shape
    heads, rows, ref = _oracle_sampled(oracle_mod, name, per_head=64)
    on = oracle_mod.norms(q, k, wl.F, wl.T, wl.w, wl.ref)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    bd = torch.empty((H, N), device=dev)
    el = torch.empty(H, dtype=torch.uint8, device=dev)
    rm = torch.full((H, N), float("nan"), device=dev)
    st = fsa.new_stats(dev)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        fsa.norms(qd, kd, plan, None, None, bd, el)
        out, lse = fsa.forward_ex(qd, kd, vd, plan, "norm_bound", bound=bd, eligible=el, rowmax=rm, stats=st)
        torch.cuda.synchronize()
    stats = fsa.read_stats(st)
    assert stats["error"] == 0
    elig = el.cpu().numpy()
    worst = on["gap_hat"].max(axis=1)
    margin = np.abs(worst - oracle_mod.DEFAULT_TAU) > 1e-3 * oracle_mod.DEFAULT_TAU
    assert np.array_equal(elig[margin], on["eligible"][margin])
    assert stats["fallback_heads"] == int((elig == 0).sum())
    # per-row tolerance from the fp32 logit error (module docstring)
    b = ref["bound"]
    vmax = float(v.abs().max())
    tol_lse = MAX_ABS + 8 * math.sqrt(D) * U32 * b
    tol_out = MAX_ABS + 8 * math.sqrt(D) * U32 * b * vmax
    o = out.cpu().double().numpy()[heads, rows]
    l = lse.cpu().double().numpy()[heads, rows]
    assert np.all(np.abs(l - ref["lse"]) <= tol_lse)
    assert np.all(np.abs(o - ref["out"]).max(axis=1) <= tol_out)
    # mean-abs over the sample, widened by the mean of the same per-row logit term
    assert np.abs(l - ref["lse"]).mean() <= MEAN_ABS + np.mean(8 * math.sqrt(D) * U32 * b)
    assert np.abs(o - ref["out"]).mean() <= MEAN_ABS + np.mean(8 * math.sqrt(D) * U32 * b * vmax)
    # underflow accounting: rows of fallback heads carry their max; the GPU flag agrees with
    # the oracle wherever the gap is not within rounding of the threshold
    rmax = rm.cpu().double().numpy()
    bnd = bd.cpu().double().numpy()
    fb = elig[heads] == 0
    gap_gpu = bnd[heads, rows] - rmax[heads, rows]
    clear = np.abs(ref["gap"] - UNDERFLOW_GAP) > 1e-3 * UNDERFLOW_GAP + 8 * math.sqrt(D) * U32 * b
    sel = fb & clear
    assert np.array_equal(gap_gpu[sel] >= UNDERFLOW_GAP, ref["underflow"][sel])
    all_fb_rows = np.repeat(elig == 0, N).reshape(H, N)
    gpu_count = int(((bnd - rmax) >= UNDERFLOW_GAP)[all_fb_rows].sum())
    assert abs(stats["underflow_rows"] - gpu_count) <= max(3, gpu_count // 1000)


# ---------------------------------------------------------------- invariances (tier 1)
def test_block_size_invariance_bitwise(dev):
    wl = WORKLOADS["sr28k"]
    q, k, v = make_qkv(2, wl.N, wl.D, seed=77)
    outs = []
    for block in (16, 48, 80, 240):
        r = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, block, "norm_bound")
        outs.append((r["out_t"].cpu(), r["lse_t"].cpu()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
def test_head_group_invariance_bitwise(dev, mode):
    wl = WORKLOADS["small"]
    q, k, v = _inputs("small")
    full = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, mode)
    half = wl.H // 2
    a = _gpu(dev, q[:half].contiguous(), k[:half].contiguous(), v[:half].contiguous(), wl.F, wl.T, wl.w, wl.ref,
             wl.block, mode)
    b = _gpu(dev, q[half:].contiguous(), k[half:].contiguous(), v[half:].contiguous(), wl.F, wl.T, wl.w, wl.ref,
             wl.block, mode)
    assert torch.equal(full["out_t"].cpu(), torch.cat([a["out_t"].cpu(), b["out_t"].cpu()]))
    assert torch.equal(full["lse_t"].cpu(), torch.cat([a["lse_t"].cpu(), b["lse_t"].cpu()]))


@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
@pytest.mark.parametrize("heads_per_chunk,pinned", [(0, True), (3, True), (1, True), (8, False)])
def test_forward_host_equals_device_bitwise(dev, mode, heads_per_chunk, pinned):
    # host tensors in, chunks of heads pipelined over three streams: same bits as the device
    # call (heads are independent); 3 heads per chunk leaves a ragged last chunk of 2
    wl = WORKLOADS["small"]
    q, k, v = _inputs("small")
    v2 = (v.float() * -0.5).to(torch.bfloat16)
    refs = [_gpu(dev, q, k, vv, wl.F, wl.T, wl.w, wl.ref, wl.block, mode) for vv in (v, v2)]
    if pinned:
        q, k, v, v2 = q.pin_memory(), k.pin_memory(), v.pin_memory(), v2.pin_memory()
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        for vv, ref in zip((v, v2), refs):  # the second call reuses the plan's device copies
            out, lse = fsa.forward_host(q, k, vv, plan, mode, heads_per_chunk=heads_per_chunk)
            torch.cuda.current_stream().synchronize()
            assert not out.is_cuda and out.is_pinned() == pinned
            assert torch.equal(out, ref["out_t"].cpu())
            assert torch.equal(lse, ref["lse_t"].cpu())


def test_forward_host_with_centred_keys_equals_device_bitwise(dev):
    # the plan option reaches the host pipeline: each chunk's norms centre its own heads' keys
    # on their own means, so the chunked result equals the one device call bit for bit
    wl = WORKLOADS["small"]
    q, k, v = make_qkv(wl.H, wl.N, wl.D, seed=44, kind="offset")
    ref = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, "norm_bound", stats=True, center_keys=True)
    assert ref["stats"]["fallback_heads"] == 0
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        plan.set_center_keys(True)
        out, lse = fsa.forward_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), plan, "norm_bound",
                                    heads_per_chunk=3)
        torch.cuda.current_stream().synchronize()
    assert torch.equal(out, ref["out_t"].cpu()) and torch.equal(lse, ref["lse_t"].cpu())


@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
@pytest.mark.parametrize("shape", [(2, 3, 1200, 64, 1, 0, 80), (4, 4, 384, 128, 1, 3, 128)])
def test_repeated_runs_are_bitwise_identical(dev, oracle_mod, shape, mode):
    # The kernel's reductions run in a fixed order, so repeated launches must agree bit for bit;
    # a race between the warps that share a row (or between softmax and MMAs) shows up here.
    H, F, T, D, w, ref, block = shape
    q, k, v = make_qkv(H, F * T, D, seed=7 + sum(shape))
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    with fsa.Plan(F, T, w, ref, block) as plan:
        runs = []
        for _ in range(6):
            out, lse = fsa.forward(qd, kd, vd, plan, mode)
            torch.cuda.synchronize()
            runs.append((out.cpu(), lse.cpu()))
    for o, l in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
    ref_res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    _check(runs[0][0].double().numpy(), runs[0][1].double().numpy(), ref_res["out"], ref_res["lse"])


def test_forced_fallback_equals_online_bitwise(dev):
    wl = WORKLOADS["small"]
    q, k, v = _inputs("small")
    fb = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, "norm_bound", tau=1e-3, stats=True)
    on = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, "online_max")
    assert fb["stats"]["fallback_heads"] == wl.H
    assert torch.equal(fb["out_t"].cpu(), on["out_t"].cpu())
    assert torch.equal(fb["lse_t"].cpu(), on["lse_t"].cpu())


def test_external_norms_match_internal(dev):
    wl = WORKLOADS["small"]
    q, k, v = _inputs("small")
    H, N, D = q.shape
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        o1, l1 = fsa.forward(qd, kd, vd, plan, "norm_bound")
        bd = torch.empty((H, N), device=dev)
        el = torch.empty(H, dtype=torch.uint8, device=dev)
        fsa.norms(qd, kd, plan, None, None, bd, el)
        o2, l2 = fsa.forward_ex(qd, kd, vd, plan, "norm_bound", bound=bd, eligible=el)
        torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bound_dominates_row_max_on_gpu(dev):
    wl = WORKLOADS["small"]
    q, k, v = _inputs("small")
    H, N, D = q.shape
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        bd = torch.empty((H, N), device=dev)
        el = torch.empty(H, dtype=torch.uint8, device=dev)
        fsa.norms(qd, kd, plan, None, None, bd, el)
        rm = torch.empty((H, N), device=dev)
        fsa.forward_ex(qd, kd, vd, plan, "online_max", bound=bd, eligible=el, rowmax=rm)
        torch.cuda.synchronize()
    b, m = bd.cpu().double().numpy(), rm.cpu().double().numpy()
    assert np.all(b >= m - 1e-5 * np.abs(b))


# ------------------------------------------------------------------- mean-centred keys
def _gpu_norms(dev, q, k, wl, center_keys, noalloc=False):
    H, N, D = q.shape
    qd, kd = q.to(dev), k.to(dev)
    qn = torch.full((H, N), -1.0, device=dev)
    km = torch.full((H, wl.F), -1.0, device=dev)
    bd = torch.full((H, N), -1.0, device=dev)
    el = torch.full((H,), 7, dtype=torch.uint8, device=dev)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        plan.set_center_keys(center_keys)
        fsa.norms(qd, kd, plan, qn, km, bd, el)
        torch.cuda.synchronize()
    return {"qnorm": qn.cpu().double().numpy(), "kmax": km.cpu().double().numpy(),
            "bound": bd.cpu().double().numpy(), "eligible": el.cpu().numpy()}


@pytest.mark.parametrize("name", ["tiny", "small", "offset"])
def test_centred_norms_parity(dev, oracle_mod, name):
    wl = WORKLOADS[name]
    q, k, _ = _inputs(name)
    H, N, D = q.shape
    on = oracle_mod.norms(q, k, wl.F, wl.T, wl.w, wl.ref, center=True)
    got = _gpu_norms(dev, q, k, wl, True)
    np.testing.assert_allclose(got["qnorm"], on["qnorm"], rtol=2e-6)
    # fp32 centring: k - mu and <q, mu> carry errors of order 2^-24 times the key and mean
    # magnitudes; the tolerance scales with c ||q|| (Kc + ||mu||)
    mu_norm = np.linalg.norm(k.double().numpy().mean(axis=1), axis=-1)  # [H], a tolerance scale only
    np.testing.assert_allclose(got["kmax"], on["kmax"], rtol=2e-5, atol=0)
    c = 1.0 / math.sqrt(D)
    scale = c * on["qnorm"] * (on["kmax"].max(axis=1) + mu_norm)[:, None]
    assert np.all(np.abs(got["bound"] - on["bound"]) <= 2e-5 * scale + 1e-6)
    worst = on["gap_hat"].max(axis=1)
    margin = np.abs(worst - oracle_mod.DEFAULT_TAU) > 1e-3 * oracle_mod.DEFAULT_TAU
    assert np.array_equal(got["eligible"][margin], on["eligible"][margin])


def test_centred_keys_make_offset_heads_eligible(dev, oracle_mod):
    # Keys that share a large per-head component: without centring most heads fail the gap
    # test and run with the running max; with centring every head takes the fixed bound.  The
    # outputs are the same attention either way (sampled rows against the oracle).
    name = "offset"
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    heads, rows, ref = _oracle_sampled(oracle_mod, name, per_head=16)
    for center, in ((False,), (True,)):
        on = oracle_mod.norms(q, k, wl.F, wl.T, wl.w, wl.ref, center=center)
        res = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, "norm_bound", stats=True,
                   center_keys=center)
        assert res["stats"]["fallback_heads"] == int((on["eligible"] == 0).sum())
        assert res["stats"]["underflow_rows"] == 0
        _check(res["out"][heads, rows], res["lse"][heads, rows], ref["out"], ref["lse"])
        if center:
            assert res["stats"]["fallback_heads"] == 0
        else:
            assert res["stats"]["fallback_heads"] >= wl.H // 2


def test_centred_bound_dominates_row_max_on_gpu(dev):
    wl = WORKLOADS["small"]
    q, k, v = make_qkv(wl.H, wl.N, wl.D, seed=41, kind="offset")
    H, N, D = q.shape
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        plan.set_center_keys(True)
        bd = torch.empty((H, N), device=dev)
        el = torch.empty(H, dtype=torch.uint8, device=dev)
        fsa.norms(qd, kd, plan, None, None, bd, el)
        rm = torch.empty((H, N), device=dev)
        fsa.forward_ex(qd, kd, vd, plan, "online_max", bound=bd, eligible=el, rowmax=rm)
        torch.cuda.synchronize()
    b, m = bd.cpu().double().numpy(), rm.cpu().double().numpy()
    # the centred bound can sit exactly at the row max, so rounding may put it a few ulps of
    # the logit magnitude below
    mag = np.abs(m) + np.abs(b) + 1.0
    assert np.all(b >= m - 1e-5 * mag)


@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
def test_centred_forward_full_parity(dev, oracle_mod, mode):
    H, F, T, D, w, ref, block = 2, 6, 128, 128, 1, 0, 64
    q, k, v = make_qkv(H, F * T, D, seed=43, kind="offset")
    exp = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    res = _gpu(dev, q, k, v, F, T, w, ref, block, mode, stats=True, center_keys=True)
    _check(res["out"], res["lse"], exp["out"], exp["lse"])
    assert res["stats"]["fallback_heads"] == 0


# ------------------------------------------------------------------------ edge shapes
EDGE = [
    # H, F, T, D, w, ref, block
    (1, 1, 16, 64, 0, 0, 16),      # one frame, smallest frame
    (2, 3, 48, 64, 0, 1, 16),      # one ragged query tile per frame, reference in the middle
    (1, 4, 384, 128, 1, 3, 128),   # three query tiles: a pair and a single; reference last
    (2, 5, 80, 128, 9, 2, 80),     # window wider than the sequence: dense attention
    (1, 2, 272, 128, 0, 1, 16),    # T = 16 * 17: key tile 16, ragged single tile of 16 rows
    (1, 3, 1200, 64, 1, 0, 80),    # D = 64 with the 28.8k frame size
]


@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
@pytest.mark.parametrize("shape", EDGE)
def test_edge_shapes_full_parity(dev, oracle_mod, shape, mode):
    H, F, T, D, w, ref, block = shape
    q, k, v = make_qkv(H, F * T, D, seed=sum(shape))
    ref_res = oracle_mod.attention_full(q, k, v, F, T, w, ref)
    res = _gpu(dev, q, k, v, F, T, w, ref, block, mode)
    _check(res["out"], res["lse"], ref_res["out"], ref_res["lse"])


@pytest.mark.parametrize("key_tile", [16, 32, 48, 64, 112, 128])
def test_key_tile_override(dev, oracle_mod, key_tile):
    # T = 1200: 32, 64, 112 and 128 leave a narrower last tile in every key run (16, 48, 80 and
    # 48 keys)
    H, F, T, D, w, ref, block = 2, 5, 1200, 128, 2, 0, 80
    q, k, v = make_qkv(H, F * T, D, seed=99)
    heads = np.repeat(np.arange(H, dtype=np.int32), 64)
    rows = np.concatenate([np.random.default_rng(h).integers(0, F * T, 64) for h in range(H)]).astype(np.int64)
    ref_res = oracle_mod.attention_rows(q, k, v, F, T, w, ref, heads, rows)
    for mode in ("norm_bound", "online_max"):
        res = _gpu(dev, q, k, v, F, T, w, ref, block, mode, key_tile=key_tile)
        _check(res["out"][heads, rows], res["lse"][heads, rows], ref_res["out"], ref_res["lse"])


def test_empty_problem_is_a_no_op(dev):
    with fsa.Plan(2, 64, 1, 0, 16) as plan:
        z = torch.empty((0, 128, 64), dtype=torch.bfloat16, device=dev)
        out = torch.empty((0, 128, 64), device=dev)
        lse = torch.empty((0, 128), device=dev)
        fsa.forward(z, z, z, plan, "norm_bound", out=out, lse=lse)
        torch.cuda.synchronize()


# ------------------------------------------------------------ norm-bound safety net
def test_loose_but_eligible_bounds_full_parity(dev, oracle_mod):
    # Keys scaled per head put the bound 20-60 nats above the row max; at tau 80 every head
    # still passes the gap test and runs with the fixed bound.  Every row against the oracle.
    # Tolerance: the logits here have a standard deviation of 3 to 4.5, not 1, so a row's weight
    # is concentrated on a few keys and the averaging behind the unit-variance tolerance is
    # gone.  Each weight enters the PV product rounded to bf16 (8 significant bits, relative
    # error at most 2^-8) while the row sum adds the unrounded weights, so
    # |out - exact| <= 2^-8 * sum_j p_j |v_j| / sum_j p_j <= 2^-8 max|v| per element, and the
    # mean error is at most 2^-8 * mean|v|.  The lse has no such term and keeps 1e-2 / 1e-3.
    # The running-max mode rounds its weights the same way and is held to the same bound.
    name = "loose"
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    ref = _oracle_full(oracle_mod, name)
    gap = ref["gap"]
    assert np.median(gap) > 25.0 and gap.max() > 50.0  # the case really is loose
    vabs = v.float().abs()
    out_max, out_mean = 2.0 ** -8 * float(vabs.max()), 2.0 ** -8 * float(vabs.mean())
    for mode in ("norm_bound", "online_max"):
        res = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, mode, tau=80.0, stats=True)
        assert res["stats"]["fallback_heads"] == 0
        assert res["stats"]["underflow_rows"] == 0
        d = np.abs(res["out"] - ref["out"])
        assert np.isfinite(res["out"]).all() and np.isfinite(res["lse"]).all()
        assert d.max() <= out_max, f"{mode}: out max-abs {d.max():.3e} > {out_max:.3e}"
        assert d.mean() <= out_mean, f"{mode}: out mean-abs {d.mean():.3e} > {out_mean:.3e}"
        _check(res["lse"], res["lse"], ref["lse"], ref["lse"])


def test_forced_bound_underflow_accounting(dev, oracle_mod):
    # Stress inputs with every head forced onto the fixed bound (tau 1e9): most rows sit more
    # than 126 ln 2 below their bound, every exp(s - b) flushes to zero and the row sum
    # underflows.  Those rows are counted by the norm-bound branch of the epilogue, which must
    # agree with the rows whose gap (bound minus the row max of a running-max pass of the same
    # kernel) reaches 126 ln 2, and with the oracle's flags on sampled rows.
    # Accuracy where it must hold: a flushed term is below 2^-126 = e^-87.3, i.e. below
    # e^(gap - 87.3) relative to the row's largest weight; with at most 10^4 keys and |v| <= 5 the
    # flushed mass stays under 1e-2 / 5 / 10^4 for gaps up to 87.3 - 15.5 = 71.8, so rows with a
    # gap of at most 70 nats meet the stress tolerance.
    H, F, T, D, w, ref_f, block = 4, 8, 1200, 128, 4, 0, 80
    q, k, v = make_qkv(H, F * T, D, seed=4, kind="stress")
    N = F * T
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    bd = torch.empty((H, N), device=dev)
    el = torch.empty(H, dtype=torch.uint8, device=dev)
    rm = torch.empty((H, N), device=dev)
    st = fsa.new_stats(dev)
    with fsa.Plan(F, T, w, ref_f, block) as plan:
        plan.set_tau(1e9)
        fsa.norms(qd, kd, plan, None, None, bd, el)
        fsa.forward_ex(qd, kd, vd, plan, "online_max", bound=bd, eligible=el, rowmax=rm)
        out, lse = fsa.forward_ex(qd, kd, vd, plan, "norm_bound", bound=bd, eligible=el, stats=st)
        torch.cuda.synchronize()
    stats = fsa.read_stats(st)
    assert stats["error"] == 0 and stats["fallback_heads"] == 0
    assert int(el.sum()) == H
    bnd, rmax = bd.cpu().double().numpy(), rm.cpu().double().numpy()
    gap_gpu = bnd - rmax
    n_under = int((gap_gpu >= UNDERFLOW_GAP).sum())
    n_band = int((np.abs(gap_gpu - UNDERFLOW_GAP) < 0.5).sum())  # rounding of the fp32 logits
    assert n_under > N  # the stress case does underflow
    assert abs(stats["underflow_rows"] - n_under) <= n_band
    # sampled rows against the oracle
    rng = np.random.default_rng(5)
    heads = np.repeat(np.arange(H, dtype=np.int32), 1000)
    rows = rng.integers(0, N, H * 1000).astype(np.int64)
    ref = oracle_mod.attention_rows(q, k, v, F, T, w, ref_f, heads, rows)
    clear = np.abs(ref["gap"] - UNDERFLOW_GAP) > 0.5
    assert np.array_equal((gap_gpu[heads, rows] >= UNDERFLOW_GAP)[clear], ref["underflow"][clear])
    ok_rows = ref["gap"] <= 70.0
    assert ok_rows.sum() >= 50
    o = out.cpu().double().numpy()[heads, rows][ok_rows]
    l = lse.cpu().double().numpy()[heads, rows][ok_rows]
    b = ref["bound"][ok_rows]
    vmax = float(v.abs().max())
    assert np.all(np.abs(l - ref["lse"][ok_rows]) <= MAX_ABS + 8 * math.sqrt(D) * U32 * b)
    assert np.all(np.abs(o - ref["out"][ok_rows]).max(axis=1) <= MAX_ABS + 8 * math.sqrt(D) * U32 * b * vmax)


# ------------------------------------------------------------------------- coverage
@pytest.mark.parametrize("name", ["tiny", "small", "sr28k"])
@pytest.mark.parametrize("mode", ["norm_bound", "online_max"])
def test_every_active_block_pair_visited_once(dev, name, mode):
    # The kernel counts the work items it finished and, per item, valid query rows times the keys
    # its tiles consumed; a complete call covers every active (query block, key block) pair of
    # the plan once: H * nnz * block^2 pairs over H * F * ceil(T / 128) items.
    wl = WORKLOADS[name]
    q, k, v = _inputs(name)
    res = _gpu(dev, q, k, v, wl.F, wl.T, wl.w, wl.ref, wl.block, mode, stats=True)
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as plan:
        nnz = plan.nnz()
    assert res["stats"]["items_done"] == wl.H * wl.F * ((wl.T + 127) // 128)
    assert res["stats"]["pairs_visited"] == wl.H * nnz * wl.block * wl.block
