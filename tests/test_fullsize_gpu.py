"""Full-size parity: the workloads at their full sizes, in the launch
configuration bench.py times, checked on sampled outputs.

The oracle computes each step's global statistics exactly over the whole
gradient buffers (copied to the host in chunks), takes its own decisions and
updates the sampled elements one by one; the GPU's outputs at those indices
must match after every step (fp32 state 1e-6 relative, abs 1e-9; 16-bit copy
1 ulp; norm 1e-5; skip and scale bit-exact).

The GPT-2-sized buffer runs its 100 steps with the clip active, and the
Llama-3-8B ZeRO-2 shard its 100 steps under a dynamic scale of 2^16 with an
overflow injected every 50 steps at a seeded index: those two steps are
skipped and halve the scale, which ends at 2^14 ("DeepSpeed tutorial" §2.2,
§3.2: skip and lower the scale on overflow; window 1000, so no growth).  The
other workloads run three steps with an overflow on the second, and so does
a flat shard of 2,200,000,007 elements (offsets past 2^31).
"""
import numpy as np
import pytest

import oracle as O
import synth
from harness import assert_state, to_np16, ulp16_diff

pytestmark = pytest.mark.gpu

CHUNK = 1 << 25


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _sample(n, seed, count):
    rng = np.random.default_rng(seed)
    tiles = np.arange(1, 50) * 2048
    parts = [rng.integers(0, n, count), np.arange(min(n, 4096)),
             np.arange(max(0, n - 4096), n), tiles - 1, tiles, tiles + 1]
    idx = np.unique(np.concatenate(parts))
    return idx[(idx >= 0) & (idx < n)]


def _chunk_stats(orc, grads, code, c0, c1):
    return orc.stats_of(orc.reduce([to_np16(g[c0:c1]) for g in grads], code))


class Run:
    """A workload as bench.Setup builds it, plus the oracle's view of a sample."""

    def __init__(self, name, extra=()):
        import torch

        import bench
        self.torch = torch
        self.s = bench.Setup(name, torch.device("cuda:0"))
        w = self.s.w
        self.code = O.FP16 if w["dtype"] == "fp16" else O.BF16
        self.nb = w["R"] * w["K"]
        self.hp = O.hparams(lr=w["lr"], weight_decay=w["wd"], max_grad_norm=w["clip"],
                            dynamic_scale=w["dynamic"], scale_window=1000)
        self.sc = O.scaler(w["scale"])
        self.orc = O.default()
        if name == "pertensor":
            self.groups = [(it["master"], it["m"], it["v"], it["param16"], it["grads"])
                           for it in self.s.items]
        else:
            self.groups = [(self.s.master, self.s.m, self.s.v, self.s.p16[0], self.s.grads)]
        # the oracle's statistics of every chunk of every group, in list order;
        # the gradients do not change between steps except for the injection
        self.chunks = []
        for gi, (_, m, _, _, grads) in enumerate(self.groups):
            n = m.numel()
            for c0 in range(0, n, CHUNK):
                c1 = min(n, c0 + CHUNK)
                self.chunks.append((gi, c0, c1, _chunk_stats(self.orc, grads, self.code, c0, c1)))
        self.samples = []
        for gi, (master, m, v, p16, _) in enumerate(self.groups):
            n = m.numel()
            idx = _sample(n, 1000 + gi, 60_000 if len(self.groups) == 1 else 2_000)
            if extra:
                ex = np.asarray(extra, dtype=np.int64)
                idx = np.unique(np.concatenate([idx, ex[(ex >= 0) & (ex < n)]]))
            ti = torch.from_numpy(idx).cuda()
            # with 16-bit masters (master None) the parameters are the state
            self.samples.append(dict(ti=ti,
                                     master=None if master is None
                                     else master[ti].cpu().numpy().copy(),
                                     m=m[ti].cpu().numpy().copy(),
                                     v=v[ti].cpu().numpy().copy(),
                                     p16=to_np16(p16[ti]) if master is None
                                     else np.zeros(idx.size, np.uint16)))

    def step(self, inject=None):
        """One GPU step and the oracle on the sample."""
        import zero_sharded_mixed_05_gb300 as z
        saved = None
        if inject is not None:
            gi, j = inject
            g = self.groups[gi][4][0]
            saved = g[j].clone()
            g[j] = float("inf")
        per = []
        for gi, c0, c1, st in self.chunks:
            if inject is not None and gi == inject[0] and c0 <= inject[1] < c1:
                st = _chunk_stats(self.orc, self.groups[gi][4], self.code, c0, c1)
            per.append(st)
        G = self.orc.fold_stats(per)
        self.s.step()
        info = z.zero_opt_last_step(self.s.h)
        d = self.orc.decide(self.hp, self.sc, G, float(self.nb))
        for smp, (_, _, _, _, grads) in zip(self.samples, self.groups):
            s = self.orc.reduce([to_np16(g[smp["ti"]]) for g in grads], self.code)
            self.orc.update(d, s, smp["master"], smp["m"], smp["v"], smp["p16"], self.code)
        if saved is not None:
            self.groups[inject[0]][4][0][inject[1]] = saved
        self.torch.cuda.synchronize()
        return info, d, G

    def check(self):
        for smp, (master, m, v, p16, _) in zip(self.samples, self.groups):
            ti = smp["ti"]
            if master is not None:
                assert_state("master", master[ti].cpu().numpy(), smp["master"])
            assert_state("m", m[ti].cpu().numpy(), smp["m"])
            assert_state("v", v[ti].cpu().numpy(), smp["v"])
            assert ulp16_diff(to_np16(p16[ti]), smp["p16"]) <= 1


def _run(name, steps=3, inject_steps=(2,), extra=()):
    """`steps` steps of workload `name`; on each step of `inject_steps` a +inf
    replaces one gradient at an index drawn from the seeded generator.
    `extra`: element indices sampled besides the seeded ones."""
    import zero_sharded_mixed_05_gb300 as z
    run = Run(name, extra)
    n0 = run.groups[0][1].numel()
    where = synth.seeded_indices(run.s.w["seed"], 99, len(inject_steps), 0, n0)
    inject_at = dict(zip(inject_steps, where))
    skipped, norms = [], []
    try:
        for step in range(1, steps + 1):
            inject = (0, inject_at[step]) if step in inject_at else None
            info, d, G = run.step(inject)
            assert info.skipped == d.skip == (1 if step in inject_at else 0)
            assert info.scale_used == d.scale_used
            assert info.t == run.sc.t
            if not d.skip:
                assert abs(info.norm - d.norm) <= 1e-5 * d.norm
                assert abs(info.sumsq - G.sumsq) <= 1e-5 * G.sumsq
                norms.append(d.norm)
            else:
                skipped.append(step)
            assert z.zero_opt_loss_scale(run.s.h, 0).as_tuple() == run.sc.as_tuple()
            run.check()
        return run.sc.as_tuple(), skipped, norms
    finally:
        z.zero_opt_destroy(run.s.h)


def test_fullsize_gpt2_100_steps():
    """GPT-2 size, 100 steps, no loss scaling, the clip active throughout."""
    (scale, clean, t, skipped_total, last), skipped, norms = _run("gpt2", 100, ())
    assert (scale, t, skipped_total, skipped) == (1.0, 100, 0, [])
    assert min(norms) > 1.0          # above max_grad_norm: every step is clipped


def test_fullsize_llama_zero2_shard_100_steps():
    """The 1,003,782,656-parameter ZeRO-2 shard for 100 steps with overflows
    on steps 50 and 100: both skipped, the scale 2^16 -> 2^15 -> 2^14."""
    (scale, clean, t, skipped_total, last), skipped, _ = _run("llama", 100, (50, 100))
    assert skipped == [50, 100]
    assert (scale, t, skipped_total, last) == (2.0 ** 14, 98, 2, 1)


def test_fullsize_fused_reduce():
    _run("fused")


def test_fullsize_per_tensor_list():
    _run("pertensor")


def test_fullsize_gpt2_low_precision_master():
    _run("gpt2_master16")


def test_fullsize_flat_shard_past_2_31_elements():
    """The GPT-2 settings on one flat bf16 shard of 2,200,000,007 elements:
    element offsets past 2^31 and a ragged last tile.  Three steps with an
    overflow on the second, sampled also around elements 2^31 and at the
    end."""
    import bench
    n = 2_200_000_007
    w = dict(bench.WORKLOADS["gpt2"])
    w["numel"] = n
    w["desc"] = w["desc"] + f" [resized to {n:,} params]"
    bench.WORKLOADS["flat_2200M"] = w
    edge = [2**31 + d for d in range(-9, 10)] + [n - 9 + d for d in range(9)]
    try:
        _run("flat_2200M", extra=edge)
    finally:
        del bench.WORKLOADS["flat_2200M"]
