"""The allocation-free statistics entry point against the handle-based one.

zero_opt_grad_stats_noalloc serves callers that may not call cudaMalloc (a
runtime whose own allocator owns all device memory, a process at its memory
limit, a path that cannot take cudaMalloc's synchronization): it keeps its
scratch in a fixed array inside the library's device image.  This test calls
it through the C ABI several times in a row -- each call reuses the scratch
left by the previous one -- and checks each result against
zero_opt_grad_stats on the same buffers, within the norm tolerance the other
parity tests use (1e-5 relative on the sum of squares; the overflow flag
exactly).  It lives in its own file so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _reference(z, grads, code, n):
    """The handle-based entry point on the same gradient buffers."""
    import torch
    dev = grads[0].device
    cfg = z.make_config(numel=n, world=1, grad_dtype=code)
    h = z.zero_opt_create(cfg)
    try:
        state = [torch.zeros(max(n, 1), device=dev) for _ in range(3)]
        p16 = torch.zeros(max(n, 1), dtype=grads[0].dtype, device=dev)
        bufs = z.make_buffers(*state, p16, grads, n_ranks=len(grads), grads_shard_local=True)
        return z.zero_opt_grad_stats(h, 0, bufs)
    finally:
        z.zero_opt_destroy(h)


def _noalloc(z, grads, code, n, out):
    import torch
    out.fill_(-1)
    z.zero_opt_grad_stats_noalloc(grads, code, n, out)
    torch.cuda.synchronize()
    raw = out.cpu().numpy()
    return float(raw.view(np.float64)[0]), int(raw.view(np.int32)[2])


def _buffers(n, nbuf, kind, dtype, seed, offset_elems=0):
    import torch
    out = []
    for b in range(nbuf):
        t = torch.empty(n + offset_elems, dtype=dtype, device="cuda:0")
        if n:
            synth.fill_gpu(t[offset_elems:], seed, 1 + b, 0, 3e-2, kind)
        out.append(t[offset_elems:])
    return out


def test_noalloc_stats_match_the_handle_path_on_consecutive_calls():
    import torch

    import zero_sharded_mixed_05_gb300 as z
    out = torch.empty(16, dtype=torch.uint8, device="cuda:0")   # one zero_opt_stats
    cases = [
        # (n, buffers, dtype, 16-byte aligned, inject an inf)
        (1_000_003, 3, "fp16", True, False),
        (777_777, 5, "bf16", False, False),
        (250_001, 2, "fp16", True, True),
        (4096, 1, "bf16", True, False),
    ]
    for i, (n, nbuf, dt, aligned, inject) in enumerate(cases):
        code = z.FP16 if dt == "fp16" else z.BF16
        kind = synth.F16 if dt == "fp16" else synth.BF16
        tdt = torch.float16 if dt == "fp16" else torch.bfloat16
        grads = _buffers(n, nbuf, kind, tdt, 0x5EED00A0 + i, 0 if aligned else 1)
        if inject:
            grads[1][n // 3] = float("inf")
        ref = _reference(z, grads, code, n)
        sumsq, nonfinite = _noalloc(z, grads, code, n, out)
        assert nonfinite == ref.nonfinite == int(inject), (i, nonfinite, ref.nonfinite)
        if not inject:
            assert abs(sumsq - ref.sumsq) <= 1e-5 * ref.sumsq, (i, sumsq, ref.sumsq)


def test_noalloc_rejects_too_many_buffers():
    import torch

    import zero_sharded_mixed_05_gb300 as z
    out = torch.empty(16, dtype=torch.uint8, device="cuda:0")
    g = torch.zeros(8, dtype=torch.float16, device="cuda:0")
    arr = (ctypes.c_void_p * 65)(*([g.data_ptr()] * 65))
    rc = z.lib().zero_opt_grad_stats_noalloc(ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
                                             65, z.FP16, 8, None, out.data_ptr())
    assert rc == z.ZERO_ERANGE
    assert b"maximum" in z.lib().zero_opt_last_error()
