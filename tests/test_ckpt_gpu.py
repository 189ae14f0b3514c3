"""Resume from sharded checkpoint files on the GPU: ten steps straight equal
five steps, a save of every rank's shard to files, a load into fresh buffers
and a fresh handle, then five more steps -- bit for bit, including the 16-bit
parameter copy rewritten from the restored master weights."""
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


def test_save_load_resume_is_bit_exact(tmp_path):
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    numel, world = 300_007, 4
    cfg = z.make_config(numel=numel, world=world, grad_dtype=z.BF16, lr=1e-3,
                        weight_decay=0.01, max_grad_norm=0.5, dynamic_scale=True,
                        init_scale=64.0, scale_window=3)
    _, _, S, P = O.shard_bounds(numel, world, 0)
    p0 = synth.normal_np(9, 0, 0, numel, 0.02, synth.F32)
    grads = []
    for s in range(10):
        g = torch.zeros(P, dtype=torch.bfloat16, device=dev)
        g[:numel] = synth.normal_torch(9, 1, numel, 0.3, synth.BF16, device=dev, offset=s * numel)
        grads.append(g)
    grads[6][1234] = float("inf")

    def fresh():
        states = []
        for r in range(world):
            b, e, _, _ = O.shard_bounds(numel, world, r)
            mst = torch.zeros(S, device=dev)
            mst[:e - b] = torch.from_numpy(p0[b:e]).to(dev)
            states.append([mst, torch.zeros(S, device=dev), torch.zeros(S, device=dev)])
        return states, torch.zeros(P, dtype=torch.bfloat16, device=dev)

    def steps(h, states, p16, lo, hi):
        for s in range(lo, hi):
            bufs = [z.make_buffers(*states[r], p16, [grads[s]]) for r in range(world)]
            G = z.zero_opt_fold_stats([z.zero_opt_grad_stats(h, r, bufs[r]) for r in range(world)])
            for r in range(world):
                z.zero_opt_step(h, r, bufs[r], global_stats=G)

    h1 = z.zero_opt_create(cfg)
    a, a16 = fresh()
    steps(h1, a, a16, 0, 10)

    h2 = z.zero_opt_create(cfg)
    b, b16 = fresh()
    steps(h2, b, b16, 0, 5)
    paths = [str(tmp_path / f"zero_rank{r}.bin") for r in range(world)]
    for r in range(world):
        z.zero_opt_save_shard(h2, r, *b[r], paths[r])
    z.zero_opt_destroy(h2)

    h3 = z.zero_opt_create(cfg)
    c, c16 = fresh()
    for x in c:
        for t in x:
            t.fill_(7.0)                       # garbage the load must overwrite
    for r in range(world):
        z.zero_opt_load_shard(h3, r, *c[r], paths[r], param16=c16)
    torch.cuda.synchronize()
    # the restored 16-bit copy is the rounding of the restored master weights
    for r in range(world):
        bb, e, _, _ = O.shard_bounds(numel, world, r)
        ref = O.f32_to_16(c[r][0][:e - bb].cpu().numpy(), O.BF16)
        assert (to_np16(c16[bb:e]) == ref).all()
    full = z.zero_opt_consolidate_fp32(paths, numel)
    cat = np.concatenate([b[r][0][:O.shard_bounds(numel, world, r)[1] - O.shard_bounds(numel, world, r)[0]].cpu().numpy()
                          for r in range(world)])
    assert (full.view(np.uint32) == cat.view(np.uint32)).all()
    steps(h3, c, c16, 5, 10)
    torch.cuda.synchronize()
    for r in range(world):
        bb, e, _, _ = O.shard_bounds(numel, world, r)
        for x, y in zip(a[r], c[r]):       # real elements; padding is never touched
            assert torch.equal(x[:e - bb].view(torch.int32), y[:e - bb].view(torch.int32))
        assert z.zero_opt_loss_scale(h1, r).as_tuple() == z.zero_opt_loss_scale(h3, r).as_tuple()
    assert torch.equal(a16.view(torch.int16), c16.view(torch.int16))
    z.zero_opt_destroy(h1)
    z.zero_opt_destroy(h3)


def test_master16_handles_have_no_shard_files(tmp_path):
    """A master16 handle keeps no fp32 masters, so shard files (which hold
    them) are refused with ZERO_ENOTSUP before any work."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    cfg = z.make_config(numel=1000, world=1, grad_dtype=z.BF16, master16=True)
    h = z.zero_opt_create(cfg)
    t = torch.zeros(1000, device="cuda:0")
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_opt_save_shard(h, 0, None, t, t, str(tmp_path / "x.zshard"))
    assert e.value.status == z.ZERO_ENOTSUP
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_opt_load_shard(h, 0, None, t, t, str(tmp_path / "x.zshard"))
    assert e.value.status == z.ZERO_ENOTSUP
    z.zero_opt_destroy(h)
