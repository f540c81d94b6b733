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
    heads, rows, ref = _oracle_sampled(oracle_mod, name, per_head=16)
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


@pytest.mark.parametrize("key_tile", [16, 32, 48, 64])
def test_key_tile_override(dev, oracle_mod, key_tile):
    # T = 1200: 32 and 64 leave a narrower last tile in every key run (16 and 48 keys)
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
