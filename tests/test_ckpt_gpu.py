"""Resume from sharded checkpoint files on the GPU, against the oracle.

Ten steps straight equal five steps, a save of every rank's shard to files, a
load into fresh buffers and a fresh handle, then five more steps -- bit for
bit, including the 16-bit parameter copy rewritten from the restored master
weights.  The oracle steps the same shards alongside: the resumed run's state
and loss scaler after ten steps match the oracle's (fp32 state 1e-6 relative,
abs 1e-9; 16-bit copy 1 ulp; scaler exactly), and the consolidation of the
five-step files (zero_to_fp32) matches the oracle's consolidation of its own
five-step shards ("DeepSpeed framework interview answer" (algomooc.com),
"训练与恢复边界": per-rank checkpoints under a fixed world size, merged into
one fp32 state dict by zero_to_fp32.py)."""
import numpy as np
import pytest

import oracle as O
import synth
from harness import assert_state, to_np16, ulp16_diff

pytestmark = pytest.mark.gpu


class OracleShards:
    """The oracle's copy of every rank's shard, stepped with the rank-order
    fold of all ranks' statistics (as the GPU side does)."""

    def __init__(self, numel, world, code, hp, scale, p0, master16=False):
        self.orc = O.default()
        self.numel, self.world, self.code, self.hp = numel, world, code, hp
        self.bounds = [O.shard_bounds(numel, world, r) for r in range(world)]
        self.sc = [O.scaler(scale) for _ in range(world)]
        self.st = []
        for b, e, _, _ in self.bounds:
            z = np.zeros(e - b, np.float32)
            if master16:
                self.st.append((None, z.copy(), z.copy(), O.f32_to_16(p0[b:e], code)))
            else:
                self.st.append((p0[b:e].copy(), z.copy(), z.copy(), np.zeros(e - b, np.uint16)))

    def step(self, g):
        """`g`: the step's gradient bit patterns (at least numel elements)."""
        parts = [g[b:e].copy() for b, e, _, _ in self.bounds]
        G = self.orc.fold_stats([self.orc.stats_of(self.orc.reduce([p], self.code))
                                 for p in parts])
        for r in range(self.world):
            self.orc.step(self.hp, self.sc[r], [parts[r]], self.code, *self.st[r], self.code,
                          1.0, G)

    def masters(self):
        """Every rank's master weights as binary32 (16-bit masters widened)."""
        return [st[0] if st[0] is not None else O.f16_to_f32(st[3], self.code)
                for st in self.st]


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
    grads, grads_np = [], []
    for s in range(10):
        g = torch.zeros(P, dtype=torch.bfloat16, device=dev)
        g[:numel] = synth.normal_torch(9, 1, numel, 0.3, synth.BF16, device=dev, offset=s * numel)
        grads.append(g)
        grads_np.append(synth.normal_np(9, 1, s * numel, numel, 0.3, synth.BF16))
    grads[6][1234] = float("inf")
    grads_np[6][1234] = 0x7F80
    hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=0.5, dynamic_scale=True,
                   scale_window=3)
    ref = OracleShards(numel, world, O.BF16, hp, 64.0, p0)
    for s in range(5):
        ref.step(grads_np[s])
    ref_full5 = O.consolidate(ref.masters(), numel)
    for s in range(5, 10):
        ref.step(grads_np[s])

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
        want16 = O.f32_to_16(c[r][0][:e - bb].cpu().numpy(), O.BF16)
        assert (to_np16(c16[bb:e]) == want16).all()
    full = z.zero_opt_consolidate_fp32(paths, numel)
    cat = np.concatenate([b[r][0][:O.shard_bounds(numel, world, r)[1] - O.shard_bounds(numel, world, r)[0]].cpu().numpy()
                          for r in range(world)])
    assert (full.view(np.uint32) == cat.view(np.uint32)).all()
    # zero_to_fp32 of the GPU's files against the oracle's merge of its shards
    assert_state("consolidated", full, ref_full5)
    steps(h3, c, c16, 5, 10)
    torch.cuda.synchronize()
    c16_np = to_np16(c16)
    for r in range(world):
        bb, e, _, _ = O.shard_bounds(numel, world, r)
        for x, y in zip(a[r], c[r]):       # real elements; padding is never touched
            assert torch.equal(x[:e - bb].view(torch.int32), y[:e - bb].view(torch.int32))
        assert z.zero_opt_loss_scale(h1, r).as_tuple() == z.zero_opt_loss_scale(h3, r).as_tuple()
        # the resumed run against the oracle's ten straight steps
        for name, x, y in zip(("master", "m", "v"), c[r], ref.st[r][:3]):
            assert_state(f"{name}[{r}]", x[:e - bb].cpu().numpy(), y)
        assert ulp16_diff(c16_np[bb:e], ref.st[r][3]) <= 1
        assert z.zero_opt_loss_scale(h3, r).as_tuple() == ref.sc[r].as_tuple()
    assert ref.sc[0].skipped_total == 1        # the overflow of step 7
    assert torch.equal(a16.view(torch.int16), c16.view(torch.int16))
    z.zero_opt_destroy(h1)
    z.zero_opt_destroy(h3)


def _m16_grads(numel, P, dt, n, dev):
    """(device gradient buffers, their host bit patterns) of n steps."""
    import torch
    kind = synth.F16 if dt == torch.float16 else synth.BF16
    out, host = [], []
    for s in range(n):
        g = torch.zeros(P, dtype=dt, device=dev)
        g[:numel] = synth.normal_torch(11, 1, numel, 0.3, kind, device=dev, offset=s * numel)
        out.append(g)
        host.append(synth.normal_np(11, 1, s * numel, numel, 0.3, kind))
    return out, host


@pytest.mark.parametrize("code", [O.BF16, O.FP16], ids=["bf16", "fp16"])
def test_master16_save_load_resume_is_bit_exact(tmp_path, code):
    """Low-precision masters: the 16-bit parameters are the masters, saved
    widened to binary32 (zero_opt_save_shard16) and restored into the 16-bit
    buffer by zero_opt_load_shard.  Eight steps straight equal four steps, a
    save of both ranks' shards, a load into fresh buffers and a fresh handle,
    and four more steps, bit for bit; consolidation gives the widened
    masters, and matches the oracle's merge of its own four-step shards; the
    resumed state after eight steps matches the oracle's."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    dt = torch.float16 if code == O.FP16 else torch.bfloat16
    numel, world = 200_003, 2
    cfg = z.make_config(numel=numel, world=world, grad_dtype=code, lr=1e-3,
                        weight_decay=0.01, max_grad_norm=0.5, dynamic_scale=True,
                        init_scale=64.0, scale_window=3, master16=True)
    _, _, S, P = O.shard_bounds(numel, world, 0)
    p0 = synth.normal_np(12, 0, 0, numel, 0.02, synth.F32)
    q0 = O.f32_to_16(p0, code)
    grads, grads_np = _m16_grads(numel, P, dt, 8, dev)
    hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=0.5, dynamic_scale=True,
                   scale_window=3)
    ref = OracleShards(numel, world, code, hp, 64.0, p0, master16=True)
    for s in range(4):
        ref.step(grads_np[s])
    ref_full4 = O.consolidate(ref.masters(), numel)
    for s in range(4, 8):
        ref.step(grads_np[s])

    def fresh():
        p16 = torch.zeros(P, dtype=dt, device=dev)
        p16[:numel] = torch.from_numpy(q0.view(np.int16).copy()).view(dt).to(dev)
        return [[torch.zeros(S, device=dev), torch.zeros(S, device=dev)]
                for _ in range(world)], p16

    def steps(h, mv, p16, lo, hi):
        for s in range(lo, hi):
            bufs = [z.make_buffers(None, *mv[r], p16, [grads[s]]) for r in range(world)]
            G = z.zero_opt_fold_stats([z.zero_opt_grad_stats(h, r, bufs[r]) for r in range(world)])
            for r in range(world):
                z.zero_opt_step(h, r, bufs[r], global_stats=G)

    h1 = z.zero_opt_create(cfg)
    a, a16 = fresh()
    steps(h1, a, a16, 0, 8)
    h2 = z.zero_opt_create(cfg)
    b, b16 = fresh()
    steps(h2, b, b16, 0, 4)
    paths = [str(tmp_path / f"m16_rank{r}.bin") for r in range(world)]
    for r in range(world):
        z.zero_opt_save_shard16(h2, r, b16, *b[r], paths[r])
    # consolidation: the full masters, widened exactly
    full = z.zero_opt_consolidate_fp32(paths, numel)
    assert (full.view(np.uint32) == O.f16_to_f32(to_np16(b16[:numel]), code).view(np.uint32)).all()
    assert_state("consolidated", full, ref_full4)
    z.zero_opt_destroy(h2)
    h3 = z.zero_opt_create(cfg)
    c, c16 = fresh()
    c16.fill_(3.0)                              # garbage the load must overwrite
    for x in c:
        for t in x:
            t.fill_(7.0)
    for r in range(world):
        z.zero_opt_load_shard(h3, r, None, *c[r], paths[r], param16=c16)
    torch.cuda.synchronize()
    assert torch.equal(b16[:numel].view(torch.int16), c16[:numel].view(torch.int16))
    steps(h3, c, c16, 4, 8)
    torch.cuda.synchronize()
    c16_np = to_np16(c16)
    for r in range(world):
        bb, e, _, _ = O.shard_bounds(numel, world, r)
        for x, y in zip(a[r], c[r]):
            assert torch.equal(x[:e - bb].view(torch.int32), y[:e - bb].view(torch.int32))
        assert z.zero_opt_loss_scale(h1, r).as_tuple() == z.zero_opt_loss_scale(h3, r).as_tuple()
        for name, x, y in zip(("m", "v"), c[r], ref.st[r][1:3]):
            assert_state(f"{name}[{r}]", x[:e - bb].cpu().numpy(), y)
        assert ulp16_diff(c16_np[bb:e], ref.st[r][3]) <= 1
        assert z.zero_opt_loss_scale(h3, r).as_tuple() == ref.sc[r].as_tuple()
    assert torch.equal(a16[:numel].view(torch.int16), c16[:numel].view(torch.int16))
    z.zero_opt_destroy(h1)
    z.zero_opt_destroy(h3)


@pytest.mark.parametrize("code", [O.BF16, O.FP16], ids=["bf16", "fp16"])
def test_master16_shard_file_round_trips_every_pattern(tmp_path, code):
    """All 65536 16-bit patterns as masters (zeros, subnormals, infinities,
    NaNs with their payloads) come back bit for bit through a shard file."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    dt = torch.float16 if code == O.FP16 else torch.bfloat16
    n = 65536
    cfg = z.make_config(numel=n, world=1, grad_dtype=code, master16=True)
    h = z.zero_opt_create(cfg)
    pats = torch.arange(n, dtype=torch.int32).to(torch.int16).view(dt).to(dev)
    m = torch.from_numpy(synth.normal_np(13, 0, 0, n, 1e-3, synth.F32)).to(dev)
    v = torch.from_numpy(np.abs(synth.normal_np(13, 1, 0, n, 1e-6, synth.F32))).to(dev)
    path = str(tmp_path / "pats.bin")
    z.zero_opt_save_shard16(h, 0, pats, m, v, path)
    q = torch.zeros(n, dtype=dt, device=dev)
    m2, v2 = torch.zeros_like(m), torch.zeros_like(v)
    z.zero_opt_load_shard(h, 0, None, m2, v2, path, param16=q)
    torch.cuda.synchronize()
    assert torch.equal(q.view(torch.int16), pats.view(torch.int16))
    assert torch.equal(m2.view(torch.int32), m.view(torch.int32))
    assert torch.equal(v2.view(torch.int32), v.view(torch.int32))
    z.zero_opt_destroy(h)


def test_fp32_shard_file_into_low_precision_masters(tmp_path):
    """A shard file of fp32 masters loaded by a master16 handle: the 16-bit
    masters are the fp32 values rounded to nearest even (the oracle's cast)."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n = 100_003
    p = synth.normal_np(14, 0, 0, n, 0.02, synth.F32)
    path = str(tmp_path / "fp32.bin")
    hf = z.zero_opt_create(z.make_config(numel=n, world=1, grad_dtype=z.BF16))
    t = lambda a: torch.from_numpy(a).to(dev)  # noqa: E731
    z.zero_opt_save_shard(hf, 0, t(p), t(np.zeros(n, np.float32)), t(np.zeros(n, np.float32)), path)
    z.zero_opt_destroy(hf)
    h = z.zero_opt_create(z.make_config(numel=n, world=1, grad_dtype=z.BF16, master16=True))
    q = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    z.zero_opt_load_shard(h, 0, None, m, v, path, param16=q)
    torch.cuda.synchronize()
    assert (to_np16(q) == O.f32_to_16(p, O.BF16)).all()
    z.zero_opt_destroy(h)


def test_shard_file_calls_check_the_master_mode(tmp_path):
    """zero_opt_save_shard refuses a master16 handle (its masters are the
    16-bit parameters: ZERO_ENOTSUP), zero_opt_save_shard16 a handle with fp32
    masters (ZERO_EINVAL), and a master16 load needs the 16-bit buffer."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    t = torch.zeros(1000, device="cuda:0")
    q = torch.zeros(1000, dtype=torch.bfloat16, device="cuda:0")
    h16 = z.zero_opt_create(z.make_config(numel=1000, world=1, grad_dtype=z.BF16, master16=True))
    h32 = z.zero_opt_create(z.make_config(numel=1000, world=1, grad_dtype=z.BF16))
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_opt_save_shard(h16, 0, None, t, t, str(tmp_path / "x.bin"))
    assert e.value.status == z.ZERO_ENOTSUP
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_opt_save_shard16(h32, 0, q, t, t, str(tmp_path / "x.bin"))
    assert e.value.status == z.ZERO_EINVAL
    z.zero_opt_save_shard16(h16, 0, q, t, t, str(tmp_path / "y.bin"))
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_opt_load_shard(h16, 0, None, t, t, str(tmp_path / "y.bin"))
    assert e.value.status == z.ZERO_EINVAL
    z.zero_opt_destroy(h16)
    z.zero_opt_destroy(h32)
