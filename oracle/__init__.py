"""Test infrastructure only: the fp64 CPU oracle for frame-structured sparse attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The CUDA library shares no code with it and never calls it.

The arithmetic lives in ``fsa_oracle.c`` (plain C, fp64, pthreads); this module
compiles it with gcc into ``oracle/_build/liboracle.so`` and marshals numpy arrays.
Inputs are bf16 tensors passed as their raw 16-bit patterns, so the oracle sees
exactly the values the GPU sees.

Method source: "HeyGen toi uu hoa mo hinh Avatar IV tren Google Cloud Trillium TPU"
(aihot.vn), sections "Xoa bo mat na" (frame mask, Fig. 3) and "Giai phong Softmax"
(norm-bound softmax, Fig. 4).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fsa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Row underflow threshold: exp(b - m) below the smallest normal fp32 (2^-126) means
# every exp(s - b) of the row underflows in fp32.  Reading of the pages' "pushes the
# exponentials toward underflow" (aihot.vn page, "Giai phong Softmax").
UNDERFLOW_GAP = 126.0 * math.log(2.0)

# Eligibility threshold on the gap upper bound, in nats.  The pages give no number;
# this is a tunable of this build ("parity unpinned").
DEFAULT_TAU = 64.0


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE fp64 semantics)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_key_frame_allowed.argtypes = [i32] * 5
            lib.oracle_key_frame_allowed.restype = i32
            lib.oracle_frame_set_size.argtypes = [i32] * 4
            lib.oracle_frame_set_size.restype = i32
            lib.oracle_plan.argtypes = [i32] * 5 + [vp, vp, i64, i32]
            lib.oracle_plan.restype = i64
            lib.oracle_attention_rows.argtypes = ([vp] * 3 + [i32] * 6 + [dbl, i64, vp, vp]
                                                  + [vp] * 6 + [i32])
            lib.oracle_attention_rows.restype = i32
            lib.oracle_norms.argtypes = [vp] * 2 + [i32] * 6 + [dbl, dbl, i32] + [vp] * 5
            lib.oracle_norms.restype = i32
            lib.oracle_prep_rows.argtypes = [vp, vp, i64] + [i32] * 3 + [dbl, dbl, i64] + [vp] * 4 + [i32]
            lib.oracle_prep_rows.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits(x) -> np.ndarray:
    """Raw bf16 bit patterns as a C-contiguous uint16 numpy array.

    Accepts a torch bf16 tensor (CPU) or a uint16 numpy array.
    """
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # local: the oracle itself needs only numpy

    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def default_threads() -> int:
    return os.cpu_count() or 1


def key_frame_allowed(F: int, w: int, ref: int, fq: int, fk: int) -> bool:
    return bool(_load().oracle_key_frame_allowed(F, w, ref, fq, fk))


def frame_set_size(F: int, w: int, ref: int, fq: int) -> int:
    return int(_load().oracle_frame_set_size(F, w, ref, fq))


def active_frame_pairs(F: int, w: int, ref: int) -> int:
    """Sum over query frames of the number of key frames attended."""
    return sum(frame_set_size(F, w, ref, f) for f in range(F))


def plan(F: int, T: int, w: int, ref: int, block: int, nthreads: int | None = None):
    """Block CSR (row_ptr int32[N/B+1], col_idx int32[nnz]) by exhaustive enumeration."""
    N = F * T
    if block <= 0 or N % block:
        raise ValueError("block must divide F*T")
    nb = N // block
    row_ptr = np.zeros(nb + 1, dtype=np.int32)
    cap = nb * nb
    col_idx = np.zeros(max(cap, 1), dtype=np.int32)
    rc = _load().oracle_plan(F, T, w, ref, block, _ptr(row_ptr), _ptr(col_idx), cap,
                             nthreads or default_threads())
    if rc == -2:
        raise ValueError("partial block: block size does not tile the frames")
    if rc < 0:
        raise ValueError(f"oracle_plan failed ({rc})")
    return row_ptr, col_idx[:rc].copy()


def attention_rows(q, k, v, F: int, T: int, w: int, ref: int, heads, rows,
                   scale: float | None = None, nthreads: int | None = None) -> dict:
    """Dense masked fp64 attention for the listed (head, row) pairs.

    q, k, v: bf16 [H][N][D] (torch CPU tensors or uint16 bit arrays of that shape).
    Returns a dict of fp64 arrays: out [R][D], lse [R], rowmax [R], bound [R],
    out_bound [R][D], lse_bound [R], gap [R] (= bound - rowmax) and underflow [R]
    (gap >= 126 ln 2).
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    H, N, D = qb.shape
    assert N == F * T and kb.shape == qb.shape and vb.shape == qb.shape
    heads = np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = heads.shape[0]
    assert rows.shape[0] == R
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    res = {name: np.zeros((R, D) if name in ("out", "out_bound") else R, dtype=np.float64)
           for name in ("out", "lse", "rowmax", "bound", "out_bound", "lse_bound")}
    rc = _load().oracle_attention_rows(
        _ptr(qb), _ptr(kb), _ptr(vb), H, F, T, D, w, ref, float(scale), R, _ptr(heads), _ptr(rows),
        _ptr(res["out"]), _ptr(res["lse"]), _ptr(res["rowmax"]), _ptr(res["bound"]),
        _ptr(res["out_bound"]), _ptr(res["lse_bound"]), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_attention_rows: bad arguments")
    res["gap"] = res["bound"] - res["rowmax"]
    res["underflow"] = res["gap"] >= UNDERFLOW_GAP
    return res


def attention_full(q, k, v, F: int, T: int, w: int, ref: int, scale: float | None = None,
                   nthreads: int | None = None) -> dict:
    """Every row of every head; results reshaped to [H][N][...]."""
    H, N, D = tuple(q.shape)
    heads = np.repeat(np.arange(H, dtype=np.int32), N)
    rows = np.tile(np.arange(N, dtype=np.int64), H)
    res = attention_rows(q, k, v, F, T, w, ref, heads, rows, scale, nthreads)
    for name in list(res):
        a = res[name]
        res[name] = a.reshape((H, N, D) if a.ndim == 2 else (H, N))
    return res


def norms(q, k, F: int, T: int, w: int, ref: int, scale: float | None = None,
          tau: float = DEFAULT_TAU, center: bool = False) -> dict:
    """Per-row norms, per-frame max key norms, row bounds, gap upper bounds, eligibility.

    center=True measures key norms about the head's mean key and adds c <q, mu> back
    into the bound (mean-centred keys)."""
    qb, kb = _bits(q), _bits(k)
    H, N, D = qb.shape
    assert N == F * T and kb.shape == qb.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    res = {"qnorm": np.zeros((H, N)), "kmax": np.zeros((H, F)), "bound": np.zeros((H, N)),
           "gap_hat": np.zeros((H, N)), "eligible": np.zeros(H, dtype=np.uint8)}
    rc = _load().oracle_norms(_ptr(qb), _ptr(kb), H, F, T, D, w, ref, float(scale), float(tau), int(bool(center)),
                              _ptr(res["qnorm"]), _ptr(res["kmax"]), _ptr(res["bound"]),
                              _ptr(res["gap_hat"]), _ptr(res["eligible"]))
    if rc != 0:
        raise ValueError("oracle_norms: bad arguments")
    return res


PREP_EPS = 1e-6       # RMS-norm epsilon (the pages give none)
PREP_ROPE_BASE = 10000.0


def prep_rows(x, w, H: int, D: int, rows, eps: float = PREP_EPS, base: float = PREP_ROPE_BASE,
              nthreads: int | None = None) -> dict:
    """RMS norm, QKV projection, rotary embedding of q and k, for the listed token rows.

    x: bf16 [N][d_model]; w: bf16 [3 H D][d_model] (q rows, then k, then v, head-major).
    Returns fp64 q, k, v of shape [R][H][D]."""
    xb, wb = _bits(x), _bits(w)
    N, dm = xb.shape
    assert wb.shape == (3 * H * D, dm)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = rows.shape[0]
    res = {name: np.zeros((R, H, D)) for name in ("q", "k", "v")}
    rc = _load().oracle_prep_rows(_ptr(xb), _ptr(wb), N, dm, H, D, float(eps), float(base), R, _ptr(rows),
                                  _ptr(res["q"]), _ptr(res["k"]), _ptr(res["v"]), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_prep_rows: bad arguments")
    return res


def prep_full(x, w, H: int, D: int, eps: float = PREP_EPS, base: float = PREP_ROPE_BASE) -> dict:
    """Every token row; q, k, v as fp64 [H][N][D] (the attention's layout)."""
    N = tuple(x.shape)[0]
    res = prep_rows(x, w, H, D, np.arange(N, dtype=np.int64), eps, base)
    return {name: np.ascontiguousarray(a.transpose(1, 0, 2)) for name, a in res.items()}


def active_flops(F: int, T: int, w: int, ref: int, H: int, D: int) -> int:
    """QK^T plus PV multiply-adds over active frame pairs only: 4 D T^2 pairs H."""
    return 4 * D * T * T * active_frame_pairs(F, w, ref) * H
