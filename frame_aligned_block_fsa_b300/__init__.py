"""Frame-aligned block-sparse attention with a norm-bound softmax, for B300 (sm_103a).

Public API (thin wrappers over the C ABI in include/fsa.h; every step runs in libfsa.so):

    plan = Plan(F, T, w, ref, block)           # fsa_plan
    norms(q, k, plan, qnorm, kmax, bound, eligible)   # fsa_norms
    out, lse = forward(q, k, v, plan, mode)    # fsa_forward, mode "norm_bound" | "online_max"
    forward_ex(...)                            # fsa_forward_ex
    out, lse = forward_host(q, k, v, plan)     # fsa_forward_host (host tensors, overlapped copies)
    q, k, v = prep(x, w, plan, H, ...)         # fsa_prep (RMS norm, QKV projection, rotary, packing, norms)

The library is loaded lazily on first use; importing the package needs no GPU.
"""
from ._lib import (FSA_ERR_CUDA, FSA_ERR_INVALID_ARG, FSA_ERR_SCRATCH_LIMIT, FSA_ERR_TIMEOUT,  # noqa: F401
                   FSA_ERR_UNSUPPORTED, FSA_OK,
                   FsaError, Plan, forward, forward_ex, forward_host, forward_masked, load, new_stats, norms, norms_noalloc, prep,
                   read_stats,
                   selftest_grid_timeout, selftest_wait_timeout, status_string)

__all__ = ["Plan", "norms", "norms_noalloc", "forward", "forward_ex", "forward_host", "forward_masked", "prep",
           "new_stats",
           "read_stats",
           "selftest_wait_timeout", "selftest_grid_timeout",
           "status_string", "load", "FsaError"]
