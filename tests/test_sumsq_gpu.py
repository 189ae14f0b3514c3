"""The sum of squares of a single gradient buffer over a wide range of
magnitudes, held to far more than the parity bar.

Pass 1 squares each converted 16-bit gradient exactly in binary32 and adds the
squares into pairs of binary32 words per thread. The addition is TwoSum, or
Fast2Sum where the kernel has shown that the running sum is at least every
square of the block. Both are error-free, and their error terms are equal.
Each CTA then sums its threads' pairs in binary32-pair arithmetic and rounds
the result once to binary64 (in binary64 throughout when one of its values
took the binary64 path), and the CTAs' partials are folded in binary64 in a
fixed order.  The total is therefore within about 1e-13 of the exact sum,
relative. The oracle computes it to within one binary64 rounding.  On gradients whose magnitudes span about
2^±20 the two must agree to 5e-12 relative. That is seven orders tighter
than the 1e-5 of the parity tests. It is also tight enough to fail if
Fast2Sum is used where its condition does not hold: that error is about
1e-10 on these inputs.

Shapes: 3,000,017 elements (chunks of 4 tiles, a ragged tail reduced from
global memory) in bf16 and fp16, 409,600,013 bf16 elements (200,001
tiles: chunks of 8), and 1,000,003 elements in bf16 and fp16 (a grid
short of one chunk per CTA, with a thread straddling the end of the run).  In the bf16 cases every millionth value is also pushed
above 2^50, out of the binary32 fast range, so that its block takes the
binary64 path and its CTA sums its partial in binary64; the fp16 cases keep
every CTA on the binary32-pair path.
"""
import numpy as np
import pytest

import oracle as O
import synth
from harness import to_np16

pytestmark = pytest.mark.gpu

SEED = 0x5EED0B00
CHUNK = 1 << 25
TOL = 5e-12


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _wide_gradients(n, code, span):
    """Seeded N(0, 1) values times 2^k, k uniform in [-span, span] (in
    binary32, then rounded to the 16-bit type)."""
    import torch
    dt = torch.float16 if code == O.FP16 else torch.bfloat16
    kind = synth.F16 if code == O.FP16 else synth.BF16
    g = torch.empty(n, dtype=dt, device="cuda")
    synth.fill_gpu(g, SEED, 1, 0, 1.0, kind)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED)
    for c0 in range(0, n, CHUNK):
        c1 = min(n, c0 + CHUNK)
        k = torch.randint(-span, span + 1, (c1 - c0,), generator=gen, device="cuda")
        g[c0:c1] = (g[c0:c1].float() * torch.exp2(k.float())).to(dt)
    if code == O.BF16:
        g[::1_000_003] = (g[::1_000_003].float() * 2.0 ** 55).to(dt)
    return g


def _oracle_sumsq(g, code):
    orc = O.default()
    per = []
    for c0 in range(0, g.numel(), CHUNK):
        c1 = min(g.numel(), c0 + CHUNK)
        per.append(orc.stats_of(orc.reduce([to_np16(g[c0:c1])], code)))
    return orc.fold_stats(per)


@pytest.mark.parametrize("code,n,span", [(O.BF16, 3_000_017, 20), (O.FP16, 3_000_017, 8),
                                         (O.BF16, 409_600_013, 20),
                                         (O.BF16, 1_000_003, 20), (O.FP16, 1_000_003, 8)],
                         ids=["bf16-3M", "fp16-3M", "bf16-410M", "bf16-1M", "fp16-1M"])
def test_sumsq_wide_range(code, n, span):
    import torch

    import zero_sharded_mixed_05_gb300 as z
    g = _wide_gradients(n, code, span)
    G = _oracle_sumsq(g, code)
    assert G.nonfinite == 0 and G.sumsq > 0.0
    cfg = z.make_config(numel=n, world=1, grad_dtype=code, lr=1e-3, max_grad_norm=1.0)
    h = z.zero_opt_create(cfg)
    try:
        master = torch.zeros(n, device="cuda")
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        p16 = torch.zeros(n, dtype=g.dtype, device="cuda")
        bufs = z.make_buffers(master, m, v, p16, [g])
        st = z.zero_opt_grad_stats(h, 0, bufs)
        z.zero_opt_step(h, 0, bufs)
        info = z.zero_opt_last_step(h)
        torch.cuda.synchronize()
        for got in (st.sumsq, info.sumsq):
            rel = abs(got - G.sumsq) / G.sumsq
            assert rel <= TOL, (got, G.sumsq, rel)
        assert info.skipped == 0
    finally:
        z.zero_opt_destroy(h)
