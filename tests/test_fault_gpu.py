"""Failure detection without a GPU fault: a bounded wait is made to expire.

The bulk-copy pass 1 waits for its copies with a limit of about a second.  The
test hook leaves one copy barrier un-armed for one launch, so that wait runs
out: the step must be reported as a fault, skipped with every piece of state
(master, m, v, 16-bit copy, loss scale, counters) unchanged, and the context
must stay usable -- the next step must equal the one a fault-free run takes.
"""
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


def _setup(z, n, dev):
    import torch
    cfg = z.make_config(numel=n, world=1, grad_dtype=z.BF16, lr=1e-3, weight_decay=0.01,
                        max_grad_norm=1.0, dynamic_scale=True, init_scale=8.0)
    h = z.zero_opt_create(cfg)
    st = [torch.from_numpy(synth.normal_np(4, 0, 0, n, 0.02, synth.F32)).to(dev),
          torch.zeros(n, device=dev), torch.zeros(n, device=dev),
          torch.zeros(n, dtype=torch.bfloat16, device=dev)]
    return h, st


def test_expired_wait_is_a_reported_no_op_and_the_context_stays_usable():
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n = 4_000_000                      # several tiles per CTA
    grads = [synth.normal_torch(4, 1, n, 0.05, synth.BF16, device=dev, offset=s * n)
             for s in range(2)]
    h, st = _setup(z, n, dev)
    ref_h, ref = _setup(z, n, dev)
    z.zero_opt_step(h, 0, z.make_buffers(*st, [grads[0]]))
    z.zero_opt_step(ref_h, 0, z.make_buffers(*ref, [grads[0]]))
    torch.cuda.synchronize()
    before = [t.clone() for t in st]
    scaler_before = z.zero_opt_loss_scale(h, 0).as_tuple()

    z.zero_opt_inject_wait_fault(h)
    z.zero_opt_step(h, 0, z.make_buffers(*st, [grads[1]]))
    info = z.zero_opt_last_step(h)
    assert info.fault == 1 and info.skipped == 1
    for a, b in zip(st, before):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert z.zero_opt_loss_scale(h, 0).as_tuple() == scaler_before

    # the same step again, without the hook, equals the fault-free run's step
    z.zero_opt_step(h, 0, z.make_buffers(*st, [grads[1]]))
    z.zero_opt_step(ref_h, 0, z.make_buffers(*ref, [grads[1]]))
    torch.cuda.synchronize()
    assert z.zero_opt_last_step(h).fault == 0
    for a, b in zip(st, ref):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert z.zero_opt_loss_scale(h, 0).as_tuple() == z.zero_opt_loss_scale(ref_h, 0).as_tuple()

    # a statistics pass that faults reports an overflow, so a fold skips
    z.zero_opt_inject_wait_fault(h)
    stats = z.zero_opt_grad_stats(h, 0, z.make_buffers(*st, [grads[1]]))
    assert stats.nonfinite == 1
    z.zero_opt_destroy(h)
    z.zero_opt_destroy(ref_h)
