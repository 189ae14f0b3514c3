"""zero_opt_step captured in a CUDA graph and replayed.

After one call on the same buffers (which builds and uploads the run table),
a step issues only its two kernel launches on the caller's stream: no
allocation, no host synchronization, and the decision (skip, clip, loss scale)
stays on the device.  So it can be captured once and replayed every step.
Replaying the graph must give exactly the state of the same number of eager
steps, bit for bit, including a skipped overflow step and the loss-scale
changes.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

N = 200_003
R = 2
STEPS = 7
SEED = 0x5EED0401


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _state(z, dev):
    import torch
    cfg = z.make_config(numel=N, world=1, grad_dtype=z.FP16, lr=1e-3, weight_decay=0.01,
                        max_grad_norm=0.5, dynamic_scale=True, init_scale=1024.0,
                        scale_window=3)
    h = z.zero_opt_create(cfg)
    master = torch.from_numpy(synth.normal_np(SEED, 0, 0, N, 0.02, synth.F32)).to(dev)
    st = [master, torch.zeros(N, device=dev), torch.zeros(N, device=dev),
          torch.zeros(N, dtype=torch.float16, device=dev)]
    grads = [torch.empty(N, dtype=torch.float16, device=dev) for _ in range(R)]
    bufs = z.make_buffers(*st, grads)
    return h, st, grads, bufs


def _fill(grads, step):
    for b, g in enumerate(grads):
        synth.fill_gpu(g, SEED, 1 + b, step * N, 1e-3 * 1024.0, synth.F16)
        if step == 4 and b == 1:
            g[12_345] = float("inf")


def test_graph_replay_equals_eager_steps():
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    he, se, ge, be = _state(z, dev)
    hg, sg, gg, bg = _state(z, dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # the first call builds the run table; both sides take it
        _fill(ge, 0)
        z.zero_opt_step(he, 0, be)
        _fill(gg, 0)
        z.zero_opt_step(hg, 0, bg)
        graph = torch.cuda.CUDAGraph()
    s.synchronize()
    with torch.cuda.graph(graph, stream=s):
        z.zero_opt_step(hg, 0, bg)
    skipped = []
    with torch.cuda.stream(s):
        for step in range(1, STEPS + 1):
            _fill(ge, step)
            z.zero_opt_step(he, 0, be)
            skipped.append(z.zero_opt_last_step(he).skipped)
            _fill(gg, step)
            graph.replay()
            assert z.zero_opt_last_step(hg).skipped == skipped[-1]
            assert z.zero_opt_loss_scale(hg, 0).as_tuple() == z.zero_opt_loss_scale(he, 0).as_tuple()
    torch.cuda.synchronize()
    assert skipped == [0, 0, 0, 1, 0, 0, 0]
    for a, b in zip(se, sg):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    z.zero_opt_destroy(he)
    z.zero_opt_destroy(hg)
