"""Host-side checks of the C ABI (no GPU): the library loads, exports every declared symbol,
builds the block plan bit-exactly like the oracle, and rejects bad arguments before any
device work."""
import ctypes
import os
import re

import numpy as np
import pytest

import frame_aligned_block_fsa_b300 as fsa
from frame_aligned_block_fsa_b300 import _lib
from frame_aligned_block_fsa_b300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fsa.h")


@pytest.fixture(scope="module")
def lib():
    from frame_aligned_block_fsa_b300 import build

    build.build()
    return fsa.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fsa_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    assert sorted(_lib.SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert fsa.status_string(code) != "unknown status"


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_plan_matches_oracle_bit_exactly(lib, oracle_mod, name):
    wl = WORKLOADS[name]
    with fsa.Plan(wl.F, wl.T, wl.w, wl.ref, wl.block) as p:
        row_ptr, col_idx = p.export()
    o_row, o_col = oracle_mod.plan(wl.F, wl.T, wl.w, wl.ref, wl.block)
    assert row_ptr.dtype == np.int32 and col_idx.dtype == np.int32
    assert np.array_equal(row_ptr, o_row)
    assert np.array_equal(col_idx, o_col)


@pytest.mark.parametrize("shape", [
    (1, 16, 0, 0, 16), (2, 32, 0, 1, 16), (6, 48, 1, 3, 16), (7, 48, 2, 6, 48), (5, 96, 9, 2, 32),
    (9, 64, 3, 4, 64), (3, 1200, 1, 1, 240), (24, 1200, 2, 0, 16),
])
def test_plan_matches_oracle_edge_shapes(lib, oracle_mod, shape):
    F, T, w, ref, B = shape
    with fsa.Plan(F, T, w, ref, B) as p:
        row_ptr, col_idx = p.export()
    o_row, o_col = oracle_mod.plan(F, T, w, ref, B)
    assert np.array_equal(row_ptr, o_row) and np.array_equal(col_idx, o_col)


def test_plan_matches_oracle_on_random_shapes(lib, oracle_mod):
    # 60 seeded shapes: frame counts 1..12, T a multiple of 16 up to 160, any window, any
    # reference frame, every block size that divides T
    rng = np.random.default_rng(2024)
    for _ in range(60):
        F = int(rng.integers(1, 13))
        T = 16 * int(rng.integers(1, 11))
        w = int(rng.integers(0, F + 2))
        ref = int(rng.integers(0, F))
        blocks = [b for b in range(16, T + 1, 16) if T % b == 0]
        B = int(blocks[rng.integers(0, len(blocks))])
        with fsa.Plan(F, T, w, ref, B) as p:
            row_ptr, col_idx = p.export()
        o_row, o_col = oracle_mod.plan(F, T, w, ref, B)
        assert np.array_equal(row_ptr, o_row) and np.array_equal(col_idx, o_col), (F, T, w, ref, B)


@pytest.mark.parametrize("args", [
    (0, 64, 1, 0, 16),      # no frames
    (4, 0, 1, 0, 16),       # no tokens
    (4, 64, -1, 0, 16),     # negative window
    (4, 64, 1, 4, 16),      # reference frame out of range
    (4, 64, 1, -1, 16),
    (4, 64, 1, 0, 24),      # block not a multiple of 16
    (4, 72, 1, 0, 16),      # block does not divide T
    (4, 64, 1, 0, 0),
    (70000, 32768, 1, 0, 16),  # F*T beyond 2^31
])
def test_plan_rejects_bad_arguments(lib, args):
    h = ctypes.c_void_p(1234)
    assert lib.fsa_plan(*args, ctypes.byref(h)) == fsa.FSA_ERR_INVALID_ARG
    assert h.value == 1234  # untouched on error
    assert lib.fsa_plan(4, 64, 1, 0, 16, None) == fsa.FSA_ERR_INVALID_ARG


def test_plan_setters_validate(lib):
    with fsa.Plan(4, 1200, 1, 0, 80) as p:
        for bad in (0.0, -1.0, float("nan")):
            assert lib.fsa_plan_set_tau(p.handle, bad) == fsa.FSA_ERR_INVALID_ARG
        assert lib.fsa_plan_set_tau(p.handle, 10.0) == fsa.FSA_OK
        for bad in (8, 24, 136, 144, -16):
            assert lib.fsa_plan_set_key_tile(p.handle, bad) == fsa.FSA_ERR_INVALID_ARG, bad
        for good in (0, 16, 48, 64, 80, 112, 128):
            assert lib.fsa_plan_set_key_tile(p.handle, good) == fsa.FSA_OK
        for bad in (-1, 2, 7):
            assert lib.fsa_plan_set_center_keys(p.handle, bad) == fsa.FSA_ERR_INVALID_ARG, bad
        for good in (1, 0):
            assert lib.fsa_plan_set_center_keys(p.handle, good) == fsa.FSA_OK
    assert lib.fsa_plan_set_center_keys(None, 1) == fsa.FSA_ERR_INVALID_ARG


def test_forward_rejects_bad_arguments_before_device_work(lib):
    # Fake, never-dereferenced, 16-byte aligned addresses: every call below must fail in
    # argument validation, before touching a device (this machine may have none).
    fake = ctypes.c_void_p(1 << 20)
    with fsa.Plan(4, 64, 1, 0, 16) as p:
        h = p.handle
        ex = lib.fsa_forward_ex
        args = lambda **kw: [kw.get("q", fake), kw.get("k", fake), kw.get("v", fake), kw.get("out", fake),
                             kw.get("lse", fake), kw.get("H", 2), kw.get("D", 64), kw.get("plan", h),
                             kw.get("mode", 0), kw.get("bound", None), kw.get("elig", None), None, None, None]
        assert ex(*args(D=96)) == fsa.FSA_ERR_UNSUPPORTED
        assert ex(*args(D=256)) == fsa.FSA_ERR_UNSUPPORTED
        assert ex(*args(mode=2)) == fsa.FSA_ERR_INVALID_ARG
        assert ex(*args(H=-1)) == fsa.FSA_ERR_INVALID_ARG
        assert ex(*args(q=None)) == fsa.FSA_ERR_INVALID_ARG
        assert ex(*args(lse=None)) == fsa.FSA_ERR_INVALID_ARG
        assert ex(*args(plan=None)) == fsa.FSA_ERR_INVALID_ARG
        assert ex(*args(q=ctypes.c_void_p((1 << 20) + 8))) == fsa.FSA_ERR_INVALID_ARG  # misaligned
        assert ex(*args(bound=fake)) == fsa.FSA_ERR_INVALID_ARG  # bound without eligibility
        assert ex(*args(H=0)) == fsa.FSA_OK  # empty problem: no work at all
        assert lib.fsa_norms(fake, fake, 2, 96, h, None, None, None, None, None) == fsa.FSA_ERR_UNSUPPORTED
        assert lib.fsa_norms(None, fake, 2, 64, h, None, None, None, None, None) == fsa.FSA_ERR_INVALID_ARG
        assert lib.fsa_norms(fake, fake, 0, 64, h, None, None, None, None, None) == fsa.FSA_OK
        assert ex(*args(H=0, q=None, k=None, v=None, out=None, lse=None)) == fsa.FSA_OK
        assert lib.fsa_forward(fake, fake, fake, fake, fake, 2, 64, h, 7, None) == fsa.FSA_ERR_INVALID_ARG
        fh = lib.fsa_forward_host
        hargs = lambda **kw: [kw.get("q", fake), kw.get("k", fake), kw.get("v", fake), kw.get("out", fake),
                              kw.get("lse", fake), kw.get("H", 2), kw.get("D", 64), kw.get("plan", h),
                              kw.get("mode", 0), kw.get("hpc", 0), None]
        assert fh(*hargs(D=96)) == fsa.FSA_ERR_UNSUPPORTED
        assert fh(*hargs(mode=3)) == fsa.FSA_ERR_INVALID_ARG
        assert fh(*hargs(hpc=-1)) == fsa.FSA_ERR_INVALID_ARG
        assert fh(*hargs(v=None)) == fsa.FSA_ERR_INVALID_ARG
        assert fh(*hargs(out=None)) == fsa.FSA_ERR_INVALID_ARG
        assert fh(*hargs(plan=None)) == fsa.FSA_ERR_INVALID_ARG
        assert fh(*hargs(H=0)) == fsa.FSA_OK
    # H * N beyond int32 row indexing
    with fsa.Plan(16, 3600, 1, 0, 144) as p:
        assert lib.fsa_forward(fake, fake, fake, fake, fake, 40000, 128, p.handle, 0, None) == \
            fsa.FSA_ERR_INVALID_ARG


def test_prep_rejects_bad_arguments_before_device_work(lib):
    # fake, never-dereferenced, 16-byte aligned addresses: every call fails in validation
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    with fsa.Plan(4, 64, 1, 0, 16) as p:
        h = p.handle

        def call(x=fake, w=fake, dm=256, H=2, D=128, q=fake, k=fake, v=fake):
            return lib.fsa_prep(x, w, dm, H, D, h, q, k, v, None, None, None, None, None, None)

        assert call(D=32) == fsa.FSA_ERR_UNSUPPORTED          # D = 64 or 128
        assert call(H=3) == fsa.FSA_ERR_UNSUPPORTED           # H D a multiple of 256 (tiles of 256 columns)
        assert call(D=64) == fsa.FSA_ERR_UNSUPPORTED          # 2 x 64 columns: half a tile
        assert call(dm=100) == fsa.FSA_ERR_INVALID_ARG        # d_model a multiple of 64
        assert call(dm=0) == fsa.FSA_ERR_INVALID_ARG
        assert call(x=None) == fsa.FSA_ERR_INVALID_ARG
        assert call(v=None) == fsa.FSA_ERR_INVALID_ARG
        assert call(w=odd) == fsa.FSA_ERR_INVALID_ARG         # 16-byte alignment
        assert call(q=odd) == fsa.FSA_ERR_INVALID_ARG
        assert call(H=0) == fsa.FSA_OK                        # empty: nothing to do
        p.set_center_keys(True)
        assert call() == fsa.FSA_ERR_UNSUPPORTED              # centred keys: norms pass only
    assert lib.fsa_prep(fake, fake, 256, 2, 128, None, fake, fake, fake, None, None, None, None, None,
                        None) == fsa.FSA_ERR_INVALID_ARG


def test_grid_selftest_rejects_bad_arguments_before_device_work():
    lib = fsa.load()
    res = (ctypes.c_int32 * 4)()
    assert lib.fsa_selftest_grid_timeout(1000, 2, 1, None, None) == fsa.FSA_ERR_INVALID_ARG
    assert lib.fsa_selftest_grid_timeout(0, 2, 1, res, None) == fsa.FSA_ERR_INVALID_ARG
    assert lib.fsa_selftest_grid_timeout(1000, 0, 1, res, None) == fsa.FSA_ERR_INVALID_ARG
    assert lib.fsa_selftest_grid_timeout(1000, 2, 2, res, None) == fsa.FSA_ERR_INVALID_ARG


def test_masked_variant_rejects_bad_block_sizes_before_device_work():
    lib = fsa.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the argument checks come first
    with fsa.Plan(4, 64, 1, 0, 16) as plan:
        for bad in (0, 64, 200, 1152, -128):
            rc = lib.fsa_forward_masked(fake, fake, fake, fake, fake, 2, 128, plan.handle, bad, None, None)
            assert rc == fsa.FSA_ERR_INVALID_ARG, bad
        rc = lib.fsa_forward_masked(fake, fake, fake, fake, fake, 2, 96, plan.handle, 128, None, None)
        assert rc == fsa.FSA_ERR_UNSUPPORTED
        # an empty problem does nothing and touches no pointer
        assert lib.fsa_forward_masked(None, None, None, None, None, 0, 128, plan.handle, 128, None, None) == fsa.FSA_OK
