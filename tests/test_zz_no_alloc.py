"""fsa_norms_noalloc: the norms entry point for callers that cannot allocate device memory.

fsa_norms grows a plan workspace with cudaMalloc; callers that own the whole device memory
budget, or that cannot take the device synchronisation of cudaMalloc/cudaFree, use
fsa_norms_noalloc instead, which keeps its scratch in a fixed array inside the library.  These
tests check that it gives bit-identical results to fsa_norms (the same kernels run in the same
order on the same inputs) on two different problems called one after the other (the second call
must not see the first call's leftovers), that it allocates no device memory, and that it
refuses problems larger than its scratch before doing any device work.

This file is named so that pytest collects it after every other test file.
"""
import ctypes

import pytest
import torch

import frame_aligned_block_fsa_b300 as fsa
from frame_aligned_block_fsa_b300.inputs import make_qkv

# (H, F, T, D, w, ref, block, seed): two problems of different shape, run back to back
CASES = [(6, 24, 1200, 128, 2, 0, 80, 31), (8, 16, 256, 64, 1, 5, 64, 32)]


def _outputs(dev, H, F, N):
    return (torch.full((H, N), -1.0, device=dev), torch.full((H, F), -1.0, device=dev),
            torch.full((H, N), -1.0, device=dev), torch.full((H,), 7, dtype=torch.uint8, device=dev))


@pytest.mark.gpu
def test_noalloc_matches_fsa_norms_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    from frame_aligned_block_fsa_b300 import build

    build.build()
    lib = fsa.load()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream()
    plans, inputs, refs = [], [], []
    for (H, F, T, D, w, ref, block, seed) in CASES:
        q, k, _ = make_qkv(H, F * T, D, seed)
        qd, kd = q.to(dev), k.to(dev)
        plan = fsa.Plan(F, T, w, ref, block)
        qn, km, bd, el = _outputs(dev, H, F, F * T)
        fsa.norms(qd, kd, plan, qn, km, bd, el, stream=stream)  # the existing entry point
        plans.append(plan)
        inputs.append((qd, kd))
        refs.append((qn, km, bd, el))
    torch.cuda.synchronize()

    # every output buffer exists before the free-memory reading, so torch allocates nothing later
    bufs = [_outputs(dev, CASES[i][0], CASES[i][1], CASES[i][1] * CASES[i][2]) for i in (0, 1, 0)]
    torch.cuda.synchronize()

    def call_noalloc(i, out):
        H, F, T, D = CASES[i][:4]
        qd, kd = inputs[i]
        qn, km, bd, el = out
        rc = lib.fsa_norms_noalloc(ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()), H, D,
                                   plans[i].handle, ctypes.c_void_p(qn.data_ptr()), ctypes.c_void_p(km.data_ptr()),
                                   ctypes.c_void_p(bd.data_ptr()), ctypes.c_void_p(el.data_ptr()),
                                   ctypes.c_void_p(stream.cuda_stream))
        assert rc == fsa.FSA_OK, fsa.status_string(rc)
        return qn, km, bd, el

    def check(i, got):
        for name, a, b in zip(("qnorm", "kmax", "bound", "eligible"), got, refs[i]):
            assert torch.equal(a, b), name

    first = call_noalloc(0, bufs[0])   # first call on this device: looks up the scratch address
    torch.cuda.synchronize()
    check(0, first)
    free_before = torch.cuda.mem_get_info()[0]
    second = call_noalloc(1, bufs[1])  # a different shape straight after
    third = call_noalloc(0, bufs[2])   # and the first problem again, over the second's leftovers
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "the no-allocation path changed free device memory"
    check(1, second)
    check(0, third)
    for p in plans:
        p.close()


def test_noalloc_rejects_problems_beyond_its_scratch_before_device_work():
    from frame_aligned_block_fsa_b300 import build

    build.build()
    lib = fsa.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    with fsa.Plan(64, 256, 1, 0, 64) as plan:
        # 80 heads x 64 frames x 128 x 4 bytes of per-frame key sums alone are 2.5 MiB: too large
        rc = lib.fsa_norms_noalloc(fake, fake, 80, 128, plan.handle, None, fake, fake, fake, None)
        assert rc == fsa.FSA_ERR_SCRATCH_LIMIT
        assert "scratch" in fsa.status_string(rc)
        rc = lib.fsa_norms_noalloc(fake, fake, 2, 128, plan.handle, None, None, fake, fake, None)
        assert rc == fsa.FSA_ERR_INVALID_ARG  # kmax is a required output
        assert lib.fsa_norms_noalloc(fake, fake, 0, 128, plan.handle, None, None, None, None, None) == fsa.FSA_OK


@pytest.mark.gpu
def test_noalloc_centred_keys_match_fsa_norms():
    # mean-centred keys through both entry points, then an uncentred call over the leftovers
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    from frame_aligned_block_fsa_b300 import build

    build.build()
    fsa.load()
    dev = torch.device("cuda:0")
    H, F, T, D, w, ref, block, seed = CASES[0]
    q, k, _ = make_qkv(H, F * T, D, seed, kind="offset")
    qd, kd = q.to(dev), k.to(dev)
    got = {}
    for center in (True, False):
        with fsa.Plan(F, T, w, ref, block) as plan:
            plan.set_center_keys(center)
            a = _outputs(dev, H, F, F * T)
            b = _outputs(dev, H, F, F * T)
            fsa.norms(qd, kd, plan, *a)
            fsa.norms_noalloc(qd, kd, plan, b[1], b[2], b[3], qnorm=b[0])
            torch.cuda.synchronize()
        for name, x, y in zip(("qnorm", "kmax", "bound", "eligible"), a, b):
            assert torch.equal(x, y), name
        got[center] = a
    # the shared key component makes the centred key norms smaller
    assert bool((got[True][1] < got[False][1]).all())
