"""The offloaded (host) step against the oracle, on the CPU.

zero_host_step runs the per-shard step on host-resident buffers with a pool of
CPU threads.  It must give what the oracle gives on the same seeded inputs:
bit-identical master, m, v and 16-bit parameters, the same skip decisions and
the same loss-scale sequence, for any thread count.  Inputs come from
``synth``; expected values only from ``oracle``.
"""
import numpy as np
import pytest

import oracle as O
import synth


@pytest.fixture(scope="module")
def z():
    from zero_sharded_mixed_05_gb300 import _build
    _build.build()
    import zero_sharded_mixed_05_gb300 as z
    z.lib()
    return z


def _kind(code):
    return synth.F16 if code == O.FP16 else synth.BF16


def run_host(z, orc, *, numel, world=1, R=1, K=1, gdtype=O.FP16, pdtype=None, steps=3,
             threads=3, lr=1e-3, wd=0.0, max_norm=0.0, dynamic=False, init_scale=1.0,
             window=1000, hysteresis=1, warmup=(0.0, 0.0, 0), sigma=1e-3, seed=0x5EED0101,
             inject=None, grads_local=False, p16_local=False, divisor=0.0,
             master=None, bias_correction=True, master16=False):
    """Step every rank of a `world`-way sharded buffer `steps` times on the host
    and with the oracle; assert bit-identical results after every step."""
    pdtype = gdtype if pdtype is None else pdtype
    inject = inject or {}
    cfg = z.make_config(numel=numel, world=world, grad_dtype=gdtype, param_dtype=pdtype, lr=lr,
                        weight_decay=wd, max_grad_norm=max_norm, dynamic_scale=dynamic,
                        init_scale=init_scale, scale_window=window, hysteresis=hysteresis,
                        warmup=warmup, bias_correction=bias_correction, master16=master16)
    hp = O.hparams(lr=lr, weight_decay=wd, max_grad_norm=max_norm, dynamic_scale=dynamic,
                   scale_window=window, hysteresis=hysteresis, warmup=warmup,
                   bias_correction=bias_correction)
    h = z.zero_host_create(cfg, threads)
    nb = R * K
    D = divisor if divisor > 0 else float(nb)
    _, _, S, P = orc.shard_bounds(numel, world, 0)
    bounds = [orc.shard_bounds(numel, world, r) for r in range(world)]
    p0 = master if master is not None else synth.normal_np(seed, 0, 0, numel, 0.02, synth.F32)
    st, ref, osc = [], [], []
    p16 = np.zeros(P, np.uint16)
    p16_loc = [np.zeros(S, np.uint16) for _ in range(world)]
    q0 = orc.f32_to_16(p0, pdtype) if master16 else None   # the 16-bit masters
    for r in range(world):
        b, e, _, _ = bounds[r]
        st.append([np.zeros(S, np.float32) for _ in range(3)])
        st[r][0][:e - b] = p0[b:e]
        ref.append([None if master16 else p0[b:e].copy(), np.zeros(e - b, np.float32),
                    np.zeros(e - b, np.float32),
                    q0[b:e].copy() if master16 else np.zeros(e - b, np.uint16)])
        osc.append(O.scaler(init_scale))
        if master16:
            p16[b:e] = q0[b:e]
            p16_loc[r][:e - b] = q0[b:e]
            st[r][0] = None
    decisions = []
    for step in range(1, steps + 1):
        scale = osc[0].scale
        grads = []
        for k in range(nb):
            g = np.zeros(P, np.uint16)
            if numel:
                g[:numel] = synth.normal_np(seed, 1 + k, step * numel, numel, sigma * scale,
                                            _kind(gdtype))
            grads.append(g)
        for (k, j, bits) in inject.get(step, []):
            grads[k][j] = bits
        bufs = []
        for r in range(world):
            b, e, _, _ = bounds[r]
            if grads_local:
                gl = []
                for g in grads:
                    loc = np.zeros(S, np.uint16)
                    loc[:e - b] = g[b:e]
                    gl.append(loc)
            else:
                gl = grads
            bufs.append(z.make_buffers(st[r][0], st[r][1], st[r][2],
                                       p16_loc[r] if p16_local else p16, gl,
                                       n_ranks=R, n_micro=K, grads_shard_local=grads_local,
                                       param16_shard_local=p16_local, divisor=divisor))
        per = [z.zero_host_grad_stats(h, r, bufs[r]) for r in range(world)]
        G = z.zero_opt_fold_stats(per) if world > 1 else None
        for r in range(world):
            z.zero_host_step(h, r, bufs[r], global_stats=G)
        info = z.zero_host_last_step(h)
        o_per = []
        for r in range(world):
            b, e, _, _ = bounds[r]
            o_per.append(orc.stats_of(orc.reduce([g[b:e].copy() for g in grads], gdtype)))
        OG = orc.fold_stats(o_per) if world > 1 else None
        for r in range(world):
            b, e, _, _ = bounds[r]
            _, dec = orc.step(hp, osc[r], [g[b:e].copy() for g in grads], gdtype, *ref[r],
                              pdtype, D, OG)
        assert info.skipped == dec.skip and info.scale_used == dec.scale_used, step
        assert info.t == osc[-1].t, step
        if not dec.skip:
            assert info.coef == dec.coef, (step, info.coef, dec.coef)
            want = OG.sumsq if OG is not None else o_per[-1].sumsq
            assert abs(info.sumsq - want) <= 1e-12 * abs(want), (step, info.sumsq, want)
        for r in range(world):
            b, e, _, _ = bounds[r]
            assert z.zero_host_loss_scale(h, r).as_tuple() == osc[r].as_tuple(), (step, r)
            for a, o, name in zip(st[r][:3], ref[r][:3], ("master", "m", "v")):
                if o is None:
                    continue
                assert (a[:e - b].view(np.uint32) == o.view(np.uint32)).all(), (step, r, name)
            got16 = p16_loc[r][:e - b] if p16_local else p16[b:e]
            assert (got16 == ref[r][3]).all(), (step, r, "param16")
            assert not st[r][1][e - b:].any()          # padding of the state untouched
        if not p16_local:
            assert not p16[numel:].any()               # padding of the parameters untouched
        decisions.append((dec.skip, dec.scale_used))
    z.zero_host_destroy(h)
    return decisions, osc


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_tiny_four_shards_with_overflow(z, orc, threads):
    """Four ranks' fp16 buffers, dynamic scale 2048, an inf at step 4: the
    overflow step is skipped everywhere and halves the scale."""
    numel = 200_003
    dec, osc = run_host(z, orc, numel=numel, world=4, R=4, gdtype=O.FP16, steps=6,
                        threads=threads, dynamic=True, init_scale=2048.0,
                        inject={4: [(2, 123_457, 0x7C00)]})
    assert [d[0] for d in dec] == [0, 0, 0, 1, 0, 0]
    assert [d[1] for d in dec] == [2048.0] * 4 + [1024.0] * 2
    assert osc[0].t == 5


def test_bf16_accumulation_clip_adamw(z, orc):
    """R=2 ranks x K=3 micro-steps of bf16 gradients, AdamW with clipping
    active (max_norm well below the norm)."""
    run_host(z, orc, numel=150_001, world=1, R=2, K=3, gdtype=O.BF16, steps=4, threads=5,
             lr=3e-4, wd=0.01, max_norm=0.05, sigma=1e-2)


def test_shard_local_buffers_and_mixed_dtypes(z, orc):
    """Shard-local gradients and 16-bit parameters, bf16 gradients with fp16
    parameters, a world whose last shard is mostly padding."""
    run_host(z, orc, numel=10_001, world=3, R=1, K=2, gdtype=O.BF16, pdtype=O.FP16, steps=3,
             threads=4, grads_local=True, p16_local=True, wd=0.1, max_norm=1.0, sigma=1e-2)


def test_hysteresis_warmup_and_window(z, orc):
    """Hysteresis 2, WarmupLR over 4 steps and a growth window of 3 clean
    steps, with overflows at steps 2, 3 and 7."""
    inj = {s: [(0, 17, 0x7E00)] for s in (2, 3, 7)}
    dec, osc = run_host(z, orc, numel=40_000, world=2, R=2, steps=10, threads=2, dynamic=True,
                        init_scale=256.0, window=3, hysteresis=2,
                        warmup=(1e-5, 1e-3, 4), inject=inj)
    assert [d[0] for d in dec] == [0, 1, 1, 0, 0, 0, 1, 0, 0, 0]


def test_cast_of_extreme_masters(z, orc):
    """lr = 0 leaves the master unchanged, so the 16-bit write-back is the
    cast of the given masters: subnormals, values around the fp16 and bf16
    maxima, ties and signed zeros must round as the oracle rounds them."""
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, 60_000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]              # finite only
    specials = np.array([0x00000000, 0x80000000, 0x477FE000, 0x477FEFFF, 0x477FF000,
                         0x477FF001, 0xC77FF000, 0x33000000, 0x33000001, 0x337FFFFF,
                         0x38800000, 0x387FFFFF, 0x7F7FFFFF, 0x7F7F8000, 0x3F808000,
                         0x3F818000, 0x00000001, 0x80800000], np.uint32)
    master = np.concatenate([specials, bits]).view(np.float32)
    for pd in (O.FP16, O.BF16):
        run_host(z, orc, numel=master.size, world=1, gdtype=O.BF16, pdtype=pd, steps=1,
                 threads=3, lr=0.0, master=master.copy(), sigma=1e-3)


def test_host_errors(z):
    cfg = z.make_config(numel=100, world=2, grad_dtype=z.FP16)
    h = z.zero_host_create(cfg, 2)
    a = [np.zeros(50, np.float32) for _ in range(3)]
    p = np.zeros(100, np.uint16)
    g = np.zeros(100, np.uint16)
    b = z.make_buffers(*a, p, [g])
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_host_step(h, 2, b)
    assert e.value.status == z.ZERO_ERANGE
    nb = z.make_buffers(*a, p, [None])
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_host_step(h, 0, nb)
    assert e.value.status == z.ZERO_EINVAL
    assert z.zero_host_threads(h) == 2
    z.zero_host_destroy(h)


@pytest.mark.parametrize("pdtype", [O.BF16, O.FP16])
def test_low_precision_master(z, orc, pdtype):
    """master16: the 16-bit parameters are the master weights (no fp32 array);
    clipping, weight decay and an overflow step included."""
    run_host(z, orc, numel=60_001, world=2, R=2, gdtype=O.BF16, pdtype=pdtype, steps=5,
             threads=3, lr=1e-3, wd=0.01, max_norm=0.5, sigma=1e-2, dynamic=True,
             init_scale=4.0, inject={3: [(1, 4242, 0x7F80)]}, master16=True)


@pytest.mark.parametrize("threads,master16", [(1, False), (5, False), (3, True)])
def test_tensor_list(z, orc, threads, master16):
    """zero_host_step_tensors on a list of ragged tensors (R*K = 2*2 fp16
    buffers, clipping): the statistics of the concatenation, every tensor
    updated with the one decision, bit-identical to the oracle; an overflow in
    the last tensor at step 2 skips the step for all of them."""
    sizes = [5000, 1, 3000, 1024, 77_777, 0, 2049]
    R, K, steps = 2, 2, 4
    cfg = z.make_config(numel=sum(sizes), world=1, grad_dtype=O.FP16, lr=1e-3,
                        weight_decay=0.01, max_grad_norm=0.4, dynamic_scale=True,
                        init_scale=8.0, master16=master16)
    hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=0.4, dynamic_scale=True,
                   scale_window=1000)
    h = z.zero_host_create(cfg, threads)
    total = sum(sizes)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    p0 = synth.normal_np(0x5EED0501, 0, 0, total, 0.02, synth.F32)
    q0 = orc.f32_to_16(p0, O.FP16)
    mine, ref = [], []
    for i, n in enumerate(sizes):
        o = offs[i]
        mine.append(dict(master=None if master16 else p0[o:o + n].copy(),
                         m=np.zeros(n, np.float32), v=np.zeros(n, np.float32),
                         p16=q0[o:o + n].copy() if master16 else np.zeros(n, np.uint16)))
        ref.append([None if master16 else p0[o:o + n].copy(), np.zeros(n, np.float32),
                    np.zeros(n, np.float32),
                    q0[o:o + n].copy() if master16 else np.zeros(n, np.uint16)])
    sc = O.scaler(8.0)
    skips = []
    for step in range(1, steps + 1):
        flat = [synth.normal_np(0x5EED0501, 1 + b, step * total, total, 1e-3 * sc.scale,
                                synth.F16) for b in range(R * K)]
        if step == 2:
            flat[3][offs[-2] + 7] = 0x7C00
        items = [dict(numel=n, master=mine[i]["master"], m=mine[i]["m"], v=mine[i]["v"],
                      param16=mine[i]["p16"],
                      grads=[fb[offs[i]:offs[i] + n] for fb in flat]) for i, n in enumerate(sizes)]
        lst = z.make_tensor_list(items, n_ranks=R, n_micro=K)
        st = z.zero_host_grad_stats_tensors(h, 0, lst)
        z.zero_host_step_tensors(h, 0, lst)
        info = z.zero_host_last_step(h)
        s_all = orc.reduce(flat, O.FP16)
        G = orc.stats_of(s_all)
        d = orc.decide(hp, sc, G, float(R * K))
        for i, n in enumerate(sizes):
            o = offs[i]
            orc.update(d, s_all[o:o + n].copy(), *ref[i], O.FP16)
        assert info.skipped == d.skip and st.nonfinite == G.nonfinite
        if not d.skip:
            assert info.coef == d.coef
        skips.append(d.skip)
        for i in range(len(sizes)):
            if not master16:
                assert (mine[i]["master"].view(np.uint32) == ref[i][0].view(np.uint32)).all()
            assert (mine[i]["m"].view(np.uint32) == ref[i][1].view(np.uint32)).all()
            assert (mine[i]["v"].view(np.uint32) == ref[i][2].view(np.uint32)).all()
            assert (mine[i]["p16"] == ref[i][3]).all()
    assert skips == [0, 1, 0, 0]
    assert z.zero_host_loss_scale(h, 0).as_tuple() == sc.as_tuple()
    z.zero_host_destroy(h)


@pytest.mark.parametrize("seed", range(12))
def test_random_configuration(z, orc, seed):
    """Seeded random layouts, buffers and optimizer settings: the host step
    stays bit-identical to the oracle."""
    rng = np.random.default_rng(1000 + seed)
    gd = int(rng.choice([O.FP16, O.BF16]))
    dynamic = bool(rng.integers(0, 2))
    numel = int(rng.choice([1, 9, 4097, 30_001, 65_536]))
    R, K = int(rng.integers(1, 4)), int(rng.integers(1, 3))
    inject = {}
    if dynamic and rng.integers(0, 2):
        inject = {int(rng.integers(1, 4)): [(int(rng.integers(0, R * K)),
                                             int(rng.integers(0, numel)),
                                             0x7C00 if gd == O.FP16 else 0x7F80)]}
    run_host(z, orc, numel=numel, world=int(rng.choice([1, 2, 3, 5])), R=R, K=K, gdtype=gd,
             pdtype=int(rng.choice([O.FP16, O.BF16])), steps=3,
             threads=int(rng.integers(1, 7)), lr=float(rng.choice([1e-4, 1e-3])),
             wd=float(rng.choice([0.0, 0.05])), max_norm=float(rng.choice([0.0, 0.1, 1.0])),
             dynamic=dynamic, init_scale=float(rng.choice([1.0, 256.0])) if dynamic else 1.0,
             window=int(rng.choice([2, 1000])), hysteresis=int(rng.choice([1, 2])),
             warmup=(0.0, 0.0, 0) if rng.integers(0, 2) else (1e-5, 1e-3, 2),
             sigma=float(rng.choice([1e-3, 1e-2])), seed=0x5EED0B00 + seed,
             inject=inject, grads_local=bool(rng.integers(0, 2)),
             p16_local=bool(rng.integers(0, 2)), master16=bool(rng.integers(0, 3) == 0),
             bias_correction=bool(rng.integers(0, 4) != 0))
