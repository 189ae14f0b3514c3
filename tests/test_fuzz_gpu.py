"""Seeded random configurations against the oracle.

Each case draws a shard layout (Ψ, N, which ranks step), the gradient buffers
(R, K, fp16/bf16, full or shard-local, misaligned or not, stashed or not),
the optimizer (lr, weight decay, clipping, bias correction, static or dynamic
scale with hysteresis and a window, WarmupLR), the master-weight mode and the
16-bit parameter type, runs
three steps on the GPU through the C ABI and on the oracle, and requires the
parity bar of the other tests: decisions and scaler state bit-exact, fp32
state within 1e-6 relative, 16-bit parameters within one ulp.  The draws
cover combinations the explicit tests leave out; the seed list is fixed, so a
failure names a reproducible case.
"""
import numpy as np
import pytest

import oracle as O
from harness import FlatCase, assert_flat_parity, run_flat

pytestmark = pytest.mark.gpu

INF = {O.FP16: 0x7C00, O.BF16: 0x7F80}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def draw(seed):
    rng = np.random.default_rng(seed)
    world = int(rng.choice([1, 2, 3, 4, 8]))
    numel = int(rng.choice([1, 7, 2049, 8191, 8193, 40_000, 123_457, 250_001]))
    ranks, micro = int(rng.integers(1, 4)), int(rng.integers(1, 3))
    gdtype = int(rng.choice([O.FP16, O.BF16]))
    dynamic = bool(rng.integers(0, 2))
    steps = 3
    inject = {}
    if dynamic and numel > 1 and rng.integers(0, 2):
        s = int(rng.integers(1, steps + 1))
        inject = {s: [(int(rng.integers(0, ranks * micro)), int(rng.integers(0, numel)),
                       INF[gdtype])]}
    master16 = bool(rng.integers(0, 4) == 0)
    case = FlatCase(
        numel=numel, world=world, ranks=ranks, micro=micro, gdtype=gdtype,
        lr=float(rng.choice([1e-4, 1e-3, 3e-3])), betas=(0.9, 0.999),
        wd=float(rng.choice([0.0, 0.01, 0.1])),
        max_norm=float(rng.choice([0.0, 0.05, 1.0])),
        bias_correction=bool(rng.integers(0, 4) != 0),
        dynamic=dynamic, init_scale=float(rng.choice([1.0, 64.0, 1024.0])) if dynamic else 1.0,
        window=int(rng.choice([2, 3, 1000])), hysteresis=int(rng.choice([1, 2])),
        warmup=(0.0, 0.0, 0) if rng.integers(0, 2) else (1e-5, 2e-3, 2),
        sigma=float(rng.choice([1e-3, 1e-2])), seed=int(0x5EED0A00 + seed), steps=steps,
        shard_local_grads=bool(rng.integers(0, 2)),
        stash=bool(ranks * micro > 4 and rng.integers(0, 2)),
        misalign=int(rng.choice([0, 0, 1, 3])), inject=inject, master16=master16)
    # drawn last, so that the earlier fields of every seed stay as they were
    case.pdtype = int(rng.choice([gdtype, gdtype, 1 - gdtype]))
    return case


@pytest.mark.parametrize("seed", range(48))
def test_random_configuration(seed):
    case = draw(seed)
    res = run_flat(case)
    assert_flat_parity(res)
