"""The allocation-free statistics entry point, against the oracle and the
handle-based entry point.

zero_opt_grad_stats_noalloc serves callers that may not call cudaMalloc (a
runtime whose own allocator owns all device memory, a process at its memory
limit, a path that cannot take cudaMalloc's synchronization): it keeps its
scratch in a fixed array inside the library's device image.  This test calls
it through the C ABI on consecutive calls -- each reuses the scratch left by
the previous one -- and checks each result against the oracle's statistics of
the same gradient bytes and against zero_opt_grad_stats on the same buffers,
within the norm tolerance the other parity tests use (1e-5 relative on the
sum of squares; the overflow flag exactly).  The cases include shards long
enough that the capped grid of 1024 CTAs walks several tiles per CTA, aligned
and not, and the device memory in use must not change across calls.  It lives
in its own file so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import synth
from harness import to_np16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _handle_path(z, grads, code, n):
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


def _oracle(grads, code, n):
    """The oracle's statistics of the binary32 sums of the same bytes."""
    orc = O.default()
    return orc.stats_of(orc.reduce([to_np16(g[:n]) for g in grads], code))


def _noalloc(z, grads, code, n, out):
    import torch
    out.fill_(0xFF)
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


CASES = [
    # (n, buffers, dtype, 16-byte aligned, inject an inf)
    (1_000_003, 3, "fp16", True, False),
    (777_777, 5, "bf16", False, False),
    (250_001, 2, "fp16", True, True),
    (4096, 1, "bf16", True, False),
    # beyond 1024 CTAs x 2048 elements: every CTA of the capped grid walks
    # two or three tiles
    (5_000_001, 2, "bf16", True, False),
    (5_000_001, 2, "fp16", False, False),
]


def test_noalloc_stats_match_the_oracle_and_the_handle_path_on_consecutive_calls():
    import torch

    import zero_sharded_mixed_05_gb300 as z
    out = torch.empty(16, dtype=torch.uint8, device="cuda:0")   # one zero_opt_stats
    inputs = []
    for i, (n, nbuf, dt, aligned, inject) in enumerate(CASES):
        code = z.FP16 if dt == "fp16" else z.BF16
        kind = synth.F16 if dt == "fp16" else synth.BF16
        tdt = torch.float16 if dt == "fp16" else torch.bfloat16
        grads = _buffers(n, nbuf, kind, tdt, 0x5EED00A0 + i, 0 if aligned else 1)
        if inject:
            grads[1][n // 3] = float("inf")
        inputs.append((n, code, grads, inject, _oracle(grads, code, n),
                       _handle_path(z, grads, code, n)))
    torch.cuda.synchronize()
    # a first call sets the entry point up on this device; after it, the calls
    # allocate nothing: neither torch's nor the CUDA driver's count of device
    # memory moves
    _noalloc(z, inputs[0][2], inputs[0][1], inputs[0][0], out)
    used0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for rep in range(2):                       # every case twice, in a row
        for i, (n, code, grads, inject, ref, hnd) in enumerate(inputs):
            sumsq, nonfinite = _noalloc(z, grads, code, n, out)
            assert nonfinite == ref.nonfinite == hnd.nonfinite == int(inject), (rep, i)
            if not inject:
                assert abs(sumsq - ref.sumsq) <= 1e-5 * ref.sumsq, (rep, i, sumsq, ref.sumsq)
                assert abs(sumsq - hnd.sumsq) <= 1e-5 * hnd.sumsq, (rep, i, sumsq, hnd.sumsq)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == used0
    assert torch.cuda.mem_get_info()[0] == free0


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


def test_noalloc_binding_checks_its_tensors():
    """The C ABI sees only pointers; the binding refuses a gradient shorter
    than n, of the other dtype or on the host, and an output under 16 bytes,
    before anything is launched."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    out = torch.empty(16, dtype=torch.uint8, device="cuda:0")
    g = torch.zeros(100, dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(ValueError):
        z.zero_opt_grad_stats_noalloc([g], z.BF16, 101, out)
    with pytest.raises(ValueError):
        z.zero_opt_grad_stats_noalloc([g], z.FP16, 100, out)
    with pytest.raises(ValueError):
        z.zero_opt_grad_stats_noalloc([g.cpu()], z.BF16, 100, out)
    with pytest.raises(ValueError):
        z.zero_opt_grad_stats_noalloc([g], z.BF16, 100, out[:8])
    with pytest.raises(ValueError):
        z.zero_opt_grad_stats_noalloc([g], z.BF16, 100, out.cpu())
    z.zero_opt_grad_stats_noalloc([g], z.BF16, 100, out)
    torch.cuda.synchronize()
    assert out.cpu().numpy().view(np.float64)[0] == 0.0
