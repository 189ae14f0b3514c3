"""Steps back to back on one stream over unchanged gradients.

Pass 1 is a programmatic dependent launch of whatever precedes it on the
stream, and pass 2 signals its dependents at its start.  So when steps follow
one another with nothing in between, the CTAs of step t+1's pass 1 may be
scheduled while step t's pass 2 still runs.  They wait, before any memory
access, for pass 2 to complete.  Twelve such steps with no host
synchronization between them must equal twelve oracle steps:
- scaler state and counters bit-exact;
- fp32 state within 1e-6 relative;
- 16-bit parameters within one ulp.
Dynamic scaling with a window of three changes the scale and the coefficient
every third step, clipping is active, and one buffer takes the bulk pass 1
and the other the multi-buffer one.
"""
import numpy as np
import pytest

import oracle as O
import synth
from harness import assert_state, to_np16, ulp16_diff

pytestmark = pytest.mark.gpu

N = 1_000_003
STEPS = 12
SEED = 0x5EED0C00


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("nbuf", [1, 3], ids=["one-buffer", "three-buffers"])
def test_back_to_back_steps_equal_the_oracle(nbuf):
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    hpk = dict(lr=1e-3, weight_decay=0.01, max_grad_norm=0.05, dynamic_scale=True,
               scale_window=3)
    cfg = z.make_config(numel=N, world=1, grad_dtype=z.BF16, init_scale=256.0, **hpk)
    hp = O.hparams(**hpk)
    orc = O.default()
    sc = O.scaler(256.0)
    p0 = synth.normal_np(SEED, 0, 0, N, 0.02, synth.F32)
    g16 = [synth.normal_np(SEED, 1 + b, 0, N, 1e-3 * 256.0, synth.BF16) for b in range(nbuf)]
    h = z.zero_opt_create(cfg)
    try:
        master = torch.from_numpy(p0.copy()).to(dev)
        m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
        p16 = torch.zeros(N, dtype=torch.bfloat16, device=dev)
        grads = [torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16).to(dev)
                 for g in g16]
        bufs = z.make_buffers(master, m, v, p16, grads)
        torch.cuda.synchronize()
        for _ in range(STEPS):
            z.zero_opt_step(h, 0, bufs)
        torch.cuda.synchronize()
        ref = (p0.copy(), np.zeros(N, np.float32), np.zeros(N, np.float32),
               np.zeros(N, np.uint16))
        skips = []
        for _ in range(STEPS):
            _, d = orc.step(hp, sc, [g.copy() for g in g16], O.BF16, *ref, O.BF16, float(nbuf))
            skips.append(d.skip)
        assert skips == [0] * STEPS
        assert z.zero_opt_loss_scale(h, 0).as_tuple() == sc.as_tuple()
        assert sc.scale == 256.0 * 2 ** (STEPS // 3)
        assert_state("master", master.cpu().numpy(), ref[0])
        assert_state("m", m.cpu().numpy(), ref[1])
        assert_state("v", v.cpu().numpy(), ref[2])
        assert ulp16_diff(to_np16(p16), ref[3]) <= 1
    finally:
        z.zero_opt_destroy(h)
