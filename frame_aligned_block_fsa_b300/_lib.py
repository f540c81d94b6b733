"""ctypes binding to libfsa.so: argument marshalling only, no arithmetic.

Every function mirrors a C entry point of include/fsa.h.  Tensors are torch tensors used
for device memory; their data pointers and the current CUDA stream are handed to the C
library, which runs every step on the GPU.  The library must exist: a missing or
unloadable libfsa.so raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfsa.so")

FSA_MODE_NORM_BOUND = 0
FSA_MODE_ONLINE_MAX = 1
MODES = {"norm_bound": FSA_MODE_NORM_BOUND, "online_max": FSA_MODE_ONLINE_MAX}

FSA_OK = 0
FSA_ERR_INVALID_ARG = -1
FSA_ERR_UNSUPPORTED = -2
FSA_ERR_CUDA = -3
FSA_ERR_TIMEOUT = -4
FSA_ERR_SCRATCH_LIMIT = -5

# Exported symbols, in the order include/fsa.h declares them.
SYMBOLS = ("fsa_plan", "fsa_plan_destroy", "fsa_plan_export", "fsa_plan_set_tau", "fsa_plan_set_key_tile",
           "fsa_plan_set_center_keys",
           "fsa_norms", "fsa_forward", "fsa_forward_ex", "fsa_forward_host", "fsa_forward_masked", "fsa_prep", "fsa_norms_noalloc",
           "fsa_last_cuda_error", "fsa_status_string", "fsa_selftest_wait_timeout",
           "fsa_selftest_grid_timeout")

_lock = threading.Lock()
_lib = None


class FsaError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {status_string(status)} ({status})")


def load():
    """Load libfsa.so (raises if it is missing: build it with `python -m frame_aligned_block_fsa_b300.build`)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing; build it with "
                                  "`python -m frame_aligned_block_fsa_b300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            i32, i64, f32, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
            lib.fsa_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
            lib.fsa_plan.restype = i32
            lib.fsa_plan_destroy.argtypes = [vp]
            lib.fsa_plan_destroy.restype = None
            lib.fsa_plan_export.argtypes = [vp, vp, vp, ctypes.POINTER(i64)]
            lib.fsa_plan_export.restype = i32
            lib.fsa_plan_set_tau.argtypes = [vp, f32]
            lib.fsa_plan_set_tau.restype = i32
            lib.fsa_plan_set_key_tile.argtypes = [vp, i32]
            lib.fsa_plan_set_key_tile.restype = i32
            lib.fsa_plan_set_center_keys.argtypes = [vp, i32]
            lib.fsa_plan_set_center_keys.restype = i32
            lib.fsa_norms.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp, vp]
            lib.fsa_norms.restype = i32
            lib.fsa_forward.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, i32, vp]
            lib.fsa_forward.restype = i32
            lib.fsa_forward_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp]
            lib.fsa_forward_ex.restype = i32
            lib.fsa_forward_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, i32, i32, vp]
            lib.fsa_forward_host.restype = i32
            lib.fsa_forward_masked.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, i32, vp, vp]
            lib.fsa_forward_masked.restype = i32
            lib.fsa_prep.argtypes = [vp, vp, i32, i32, i32, vp] + [vp] * 9
            lib.fsa_prep.restype = i32
            lib.fsa_norms_noalloc.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp, vp]
            lib.fsa_norms_noalloc.restype = i32
            lib.fsa_last_cuda_error.argtypes = []
            lib.fsa_last_cuda_error.restype = i32
            lib.fsa_status_string.argtypes = [i32]
            lib.fsa_status_string.restype = ctypes.c_char_p
            lib.fsa_selftest_wait_timeout.argtypes = [ctypes.c_longlong, ctypes.POINTER(ctypes.c_int32), vp]
            lib.fsa_selftest_wait_timeout.restype = i32
            lib.fsa_selftest_grid_timeout.argtypes = [ctypes.c_longlong, i32, i32, ctypes.POINTER(ctypes.c_int32), vp]
            lib.fsa_selftest_grid_timeout.restype = i32
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().fsa_status_string(int(status)).decode()


def _check(call: str, status: int):
    if status != FSA_OK:
        err = FsaError(call, status)
        if status == FSA_ERR_CUDA:
            code = load().fsa_last_cuda_error()
            err.cuda_error = code
            err.args = (f"{err.args[0]} [CUDA error code {code}]",)
        raise err


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """Owner of an fsa_plan_t (frame-aligned block plan + device work list + workspace)."""

    def __init__(self, F: int, T: int, w: int, ref: int, block: int):
        lib = load()
        h = ctypes.c_void_p()
        _check("fsa_plan", lib.fsa_plan(F, T, w, ref, block, ctypes.byref(h)))
        self._h = h
        self.F, self.T, self.w, self.ref, self.block = F, T, w, ref, block
        self.N = F * T

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("plan was closed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None:
            load().fsa_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def nnz(self) -> int:
        n = ctypes.c_int64()
        _check("fsa_plan_export", load().fsa_plan_export(self.handle, None, None, ctypes.byref(n)))
        return int(n.value)

    def export(self):
        """Block CSR as numpy arrays (row_ptr int32[N/block+1], col_idx int32[nnz])."""
        import numpy as np

        nnz = self.nnz()
        row_ptr = np.zeros(self.N // self.block + 1, dtype=np.int32)
        col_idx = np.zeros(max(nnz, 1), dtype=np.int32)
        n = ctypes.c_int64()
        _check("fsa_plan_export", load().fsa_plan_export(self.handle, row_ptr.ctypes.data_as(ctypes.c_void_p),
                                                         col_idx.ctypes.data_as(ctypes.c_void_p),
                                                         ctypes.byref(n)))
        return row_ptr, col_idx[:nnz]

    def set_tau(self, tau: float):
        _check("fsa_plan_set_tau", load().fsa_plan_set_tau(self.handle, float(tau)))

    def set_key_tile(self, key_tile: int):
        _check("fsa_plan_set_key_tile", load().fsa_plan_set_key_tile(self.handle, int(key_tile)))

    def set_center_keys(self, on: bool):
        _check("fsa_plan_set_center_keys", load().fsa_plan_set_center_keys(self.handle, int(on)))


def _check_qkv(plan: Plan, *ts):
    import torch

    q = ts[0]
    if q.dim() != 3:
        raise ValueError("expected [H, N, D] tensors")
    H, N, D = q.shape
    if N != plan.N:
        raise ValueError(f"sequence length {N} != plan F*T = {plan.N}")
    for t in ts:
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA bf16 tensors of one shape [H, N, D]")
    return H, N, D


def norms(q, k, plan: Plan, qnorm=None, kmax=None, bound=None, eligible=None, stream=None):
    """fsa_norms: fills the given fp32/uint8 tensors (any may be None)."""
    H, N, D = _check_qkv(plan, q, k)
    st = _stream_handle(stream)
    _check("fsa_norms", load().fsa_norms(_ptr(q), _ptr(k), H, D, plan.handle, _ptr(qnorm), _ptr(kmax),
                                         _ptr(bound), _ptr(eligible), st))


def norms_noalloc(q, k, plan: Plan, kmax, bound, eligible, qnorm=None, stream=None):
    """fsa_norms_noalloc: fsa_norms without any device allocation (fixed in-library scratch)."""
    H, N, D = _check_qkv(plan, q, k)
    st = _stream_handle(stream)
    _check("fsa_norms_noalloc", load().fsa_norms_noalloc(_ptr(q), _ptr(k), H, D, plan.handle, _ptr(qnorm),
                                                         _ptr(kmax), _ptr(bound), _ptr(eligible), st))


def forward(q, k, v, plan: Plan, mode: str = "norm_bound", out=None, lse=None, stream=None):
    """fsa_forward: returns (out fp32 [H,N,D], lse fp32 [H,N])."""
    import torch

    H, N, D = _check_qkv(plan, q, k, v)
    if out is None:
        out = torch.empty((H, N, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((H, N), dtype=torch.float32, device=q.device)
    st = _stream_handle(stream)
    _check("fsa_forward", load().fsa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), H, D,
                                             plan.handle, MODES[mode], st))
    return out, lse


def forward_host(q, k, v, plan: Plan, mode: str = "norm_bound", out=None, lse=None, heads_per_chunk: int = 0,
                 stream=None):
    """fsa_forward_host: q, k, v are host (CPU) bf16 [H, N, D] tensors, pinned for overlap.

    Returns host (out fp32 [H,N,D], lse fp32 [H,N]); they are complete once `stream` (the
    current CUDA stream by default) has been synchronised.
    """
    import torch

    q0 = q
    if q0.dim() != 3:
        raise ValueError("expected [H, N, D] tensors")
    H, N, D = q0.shape
    if N != plan.N:
        raise ValueError(f"sequence length {N} != plan F*T = {plan.N}")
    for t in (q, k, v):
        if t.shape != q0.shape or t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous host bf16 tensors of one shape [H, N, D]")
    pin = q0.is_pinned()
    if out is None:
        out = torch.empty((H, N, D), dtype=torch.float32, pin_memory=pin)
    if lse is None:
        lse = torch.empty((H, N), dtype=torch.float32, pin_memory=pin)
    if out.is_cuda or lse.is_cuda or out.dtype != torch.float32 or lse.dtype != torch.float32:
        raise ValueError("out and lse must be host fp32 tensors")
    st = _stream_handle(stream)
    _check("fsa_forward_host", load().fsa_forward_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), H, D,
                                                       plan.handle, MODES[mode], int(heads_per_chunk), st))
    return out, lse


def prep(x, w, plan: Plan, H: int, q=None, k=None, v=None, qnorm=None, kmax=None, bound=None, eligible=None,
         stats=None, stream=None):
    """fsa_prep: x bf16 [N, d_model], w bf16 [3 H D, d_model] (device; D = w rows / 3H) ->
    (q, k, v) bf16 [H, N, D], with the norms written to the given tensors (or kept in the plan)."""
    import torch

    if x.dim() != 2 or w.dim() != 2 or x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise ValueError("x and w must be 2-D bf16 tensors")
    N, dm = x.shape
    if H <= 0 or w.shape[0] % (3 * H):
        raise ValueError("w must have 3 H D rows")
    D = w.shape[0] // (3 * H)
    if N != plan.N:
        raise ValueError(f"sequence length {N} != plan F*T = {plan.N}")
    if tuple(w.shape) != (3 * H * D, dm):
        raise ValueError(f"w must be [{3 * H * D}, {dm}]")
    if not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("x and w must be contiguous")
    outs = []
    for t in (q, k, v):
        if t is None:
            t = torch.empty((H, N, D), dtype=torch.bfloat16, device=x.device)
        elif tuple(t.shape) != (H, N, D) or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"q, k, v must be contiguous bf16 [H, N, {D}]")
        outs.append(t)
    st = _stream_handle(stream)
    _check("fsa_prep", load().fsa_prep(_ptr(x), _ptr(w), dm, H, D, plan.handle, _ptr(outs[0]), _ptr(outs[1]),
                                       _ptr(outs[2]), _ptr(qnorm), _ptr(kmax), _ptr(bound), _ptr(eligible),
                                       _ptr(stats), st))
    return tuple(outs)


def new_stats(device):
    """A zeroed device fsa_stats_t (32 bytes) as an int64 tensor of 4 words."""
    import torch

    return torch.zeros(4, dtype=torch.int64, device=device)


def read_stats(stats) -> dict:
    w32 = stats.cpu().view(__import__("torch").int32)
    return {"error": int(w32[0]), "timeout_site": int(w32[1]), "fallback_heads": int(w32[2]),
            "items_done": int(w32[3]), "underflow_rows": int(stats[2].item()),
            "pairs_visited": int(stats[3].item())}


def forward_ex(q, k, v, plan: Plan, mode: str = "norm_bound", out=None, lse=None, bound=None, eligible=None,
               rowmax=None, stats=None, stream=None):
    """fsa_forward_ex: optional precomputed norms, row maxima and device statistics."""
    import torch

    H, N, D = _check_qkv(plan, q, k, v)
    if out is None:
        out = torch.empty((H, N, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((H, N), dtype=torch.float32, device=q.device)
    st = _stream_handle(stream)
    _check("fsa_forward_ex", load().fsa_forward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), H, D,
                                                   plan.handle, MODES[mode], _ptr(bound), _ptr(eligible),
                                                   _ptr(rowmax), _ptr(stats), st))
    return out, lse


def forward_masked(q, k, v, plan: Plan, block: int = 128, out=None, lse=None, stats=None, stream=None):
    """fsa_forward_masked: the masked-block comparison variant (blocks of `block` tokens over the
    padded sequence, mask predicates, window and reference passes plus a merge)."""
    import torch

    H, N, D = _check_qkv(plan, q, k, v)
    if out is None:
        out = torch.empty((H, N, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((H, N), dtype=torch.float32, device=q.device)
    _check("fsa_forward_masked", load().fsa_forward_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), H, D,
                                                           plan.handle, int(block), _ptr(stats),
                                                           _stream_handle(stream)))
    return out, lse


def selftest_wait_timeout(limit_cycles: int, stream=None) -> int:
    status = ctypes.c_int32(0)
    _check("fsa_selftest_wait_timeout",
           load().fsa_selftest_wait_timeout(int(limit_cycles), ctypes.byref(status), _stream_handle(stream)))
    return int(status.value)


def selftest_grid_timeout(limit_cycles: int, ctas: int, missing: int, stream=None) -> dict:
    """Run the bounded grid-barrier self test; returns the kernel's report."""
    res = (ctypes.c_int32 * 4)()
    _check("fsa_selftest_grid_timeout",
           load().fsa_selftest_grid_timeout(int(limit_cycles), int(ctas), int(missing), res,
                                            _stream_handle(stream)))
    return {"status": int(res[0]), "site": int(res[1]), "gave_up": int(res[2]), "arrived": int(res[3])}
