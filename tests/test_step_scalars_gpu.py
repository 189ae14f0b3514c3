"""The update scalars the host supplies with each step, against the oracle.

The host keeps each rank's Adam step counter as it expects it (one more per
stepping launch) and passes the update scalars of that step and of the seven
below it; pass 1 takes the one that matches the device's counter and computes
them itself otherwise.  These runs step without reading the scaler state in
between, so skipped steps put the host's expectation ahead of the device: up
to seven skips the candidates still cover the device's step, after that the
device's own computation takes over, until a read of the scaler state sets
the host's counter again.  WarmupLR makes every step's scalars different, and
a learning-rate change mid-run must reach the candidates.  The state must
match the oracle's (fp32 1e-6 relative, abs 1e-9; 16-bit copy 1 ulp; the
scaler exactly), as in every other parity test.
"""
import numpy as np
import pytest

import oracle as O
import synth
from harness import assert_state, to_np16, ulp16_diff

pytestmark = pytest.mark.gpu

N = 100_003
SEED = 0x5EED0601


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _run(skip_steps, steps, warmup, lr_changes, read_at=()):
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    kw = dict(weight_decay=0.01, max_grad_norm=0.5, dynamic_scale=True, scale_window=3,
              warmup=warmup)
    h = z.zero_opt_create(z.make_config(numel=N, world=1, grad_dtype=z.BF16, lr=1e-3,
                                        init_scale=256.0, **kw))
    hp = O.hparams(lr=1e-3, **kw)
    sc = O.scaler(256.0)
    orc = O.default()
    p0 = synth.normal_np(SEED, 0, 0, N, 0.02, synth.F32)
    state = [torch.from_numpy(p0).to(dev), torch.zeros(N, device=dev),
             torch.zeros(N, device=dev), torch.zeros(N, dtype=torch.bfloat16, device=dev)]
    ref = (p0.copy(), np.zeros(N, np.float32), np.zeros(N, np.float32), np.zeros(N, np.uint16))
    g = torch.empty(N, dtype=torch.bfloat16, device=dev)
    bufs = z.make_buffers(*state, [g])
    skipped = []
    try:
        for step in range(1, steps + 1):
            if step in lr_changes:
                z.zero_opt_set_lr(h, lr_changes[step])
                hp.lr = lr_changes[step]
            gn = synth.normal_np(SEED, 1, step * N, N, 1e-3 * sc.scale, synth.BF16)
            if step in skip_steps:
                gn[(step * 7919) % N] = 0x7F80                  # +inf
            g.copy_(torch.from_numpy(gn.view(np.int16)).view(torch.bfloat16))
            z.zero_opt_step(h, 0, bufs)
            _, d = orc.step(hp, sc, [gn], O.BF16, *ref, O.BF16, 1.0)
            if d.skip:
                skipped.append(step)
            if step in read_at:
                assert z.zero_opt_loss_scale(h, 0).as_tuple() == sc.as_tuple(), step
        torch.cuda.synchronize()
        assert skipped == sorted(skip_steps)
        assert z.zero_opt_loss_scale(h, 0).as_tuple() == sc.as_tuple()
        for name, x, y in zip(("master", "m", "v"), state[:3], ref[:3]):
            assert_state(name, x.cpu().numpy(), y)
        assert ulp16_diff(to_np16(state[3]), ref[3]) <= 1
    finally:
        z.zero_opt_destroy(h)


def test_unseen_skips_within_the_candidate_window():
    """Five skips, never read back: the candidates cover the device's step
    throughout."""
    _run({4, 5, 9, 14, 15}, 30, (0.0, 1e-3, 20), {})


def test_unseen_skips_beyond_the_candidate_window():
    """Ten consecutive skips, never read back: from the eighth on the device
    computes the scalars itself; a read of the scaler state afterwards puts
    the host back in step."""
    _run(set(range(3, 13)), 40, (0.0, 1e-3, 25), {}, read_at=(30,))


def test_learning_rate_changes_reach_the_candidates():
    """A constant learning rate changed twice by zero_opt_set_lr, with skips
    the host does not see."""
    _run({6, 7, 20}, 30, (0.0, 0.0, 0), {10: 3e-4, 18: 2e-3})
