"""GPU parity of the CUDA path (through the C ABI) against the oracle.

Each test runs seeded inputs shaped like one workload at a size the oracle
finishes in seconds, spanning many 2048-element tiles and a ragged tail, and
compares element by element: flags, skip decisions, the loss-scale sequence
and counters bit-exactly; fp32 master/m/v within 1e-6 relative (abs floor
1e-9); 16-bit parameters within 1 ulp; the gradient norm within 1e-5 relative.
"""
import numpy as np
import pytest

import oracle as O
import synth
from harness import (FlatCase, assert_flat_parity, assert_state, exact_fraction,
                     llama_like_shapes, run_flat, run_list, to_np16, ulp16_diff)

pytestmark = pytest.mark.gpu

INF16, NINF16, NAN16 = 0x7C00, 0xFC00, 0x7E00
INF_BF16 = 0x7F80


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


# ---------------------------------------------------------------- generator

@pytest.mark.parametrize("kind", [synth.F32, synth.F16, synth.BF16])
def test_synth_gpu_matches_numpy(kind):
    import torch
    n, off = 100_003, 777
    t = synth.normal_torch(7, 3, n, 0.37, kind, device="cuda", offset=off)
    ref = synth.normal_np(7, 3, off, n, 0.37, kind)
    got = t.cpu()
    if kind == synth.F32:
        assert (got.numpy().view(np.uint32) == ref.view(np.uint32)).all()
    else:
        assert (got.view(torch.int16).numpy().view(np.uint16) == ref).all()


# ---------------------------------------------------------------- the five workloads

def _tiny_inject():
    # +inf in one seeded rank's buffer at one seeded real index, on step 4
    r, j = synth.seeded_indices(0x5EED0001, 99, 1, 0, 4)[0], \
        synth.seeded_indices(0x5EED0001, 98, 1, 0, 1_000_003)[0]
    return {4: [(r, j, INF16)]}


def test_tiny_n4_ten_steps_with_overflow():
    """1,000,003 fp16 parameters over 4 simulated ranks (padded to 1,000,004),
    loss scale 2048, Adam lr 1e-3, +inf on step 4: skip and halve."""
    case = FlatCase(numel=1_000_003, world=4, ranks=4, gdtype=O.FP16, lr=1e-3,
                    dynamic=True, init_scale=2048.0, window=1000, sigma=1e-3,
                    steps=10, inject=_tiny_inject())
    res = run_flat(case)
    skips = [h["gpu"][0] for h in res["history"]]
    scales = [h["gpu"][1] for h in res["history"]]
    assert skips == [0, 0, 0, 1, 0, 0, 0, 0, 0, 0]
    assert scales == [2048.0] * 4 + [1024.0] * 6
    assert res["history"][-1]["gpu"][2] == 9
    # no clipping: the coefficient does not depend on the norm, so the whole
    # state must agree bit for bit
    assert_flat_parity(res, exact=True)


def test_tiny_union_of_shards_equals_unsharded():
    """Four shard steps with folded statistics give bit-identical master/m/v/
    param16 to one unsharded step over the same four full buffers."""
    base = dict(numel=1_000_003, ranks=4, gdtype=O.FP16, lr=1e-3, dynamic=True,
                init_scale=2048.0, sigma=1e-3, steps=3)
    sh = run_flat(FlatCase(world=4, **base))
    un = run_flat(FlatCase(world=1, **base))
    for i in range(4):
        cat = np.concatenate([sh["gpu"][r][i] for r in range(4)])
        assert (cat.view(np.uint8) == un["gpu"][0][i].view(np.uint8)).all(), i


def test_gpt2_like_bf16_clip():
    """bf16 gradients ~N(0, 1e-2), N=1, no loss scaling, AdamW lr 3e-4 wd 0.01,
    global-norm clip 1.0 (active every step), 30 steps; 1,000,003 parameters."""
    case = FlatCase(numel=1_000_003, world=1, gdtype=O.BF16, lr=3e-4, wd=0.01,
                    max_norm=1.0, sigma=1e-2, steps=30, seed=0x5EED0002)
    res = run_flat(case, check_every_step=False)
    assert all(h["gpu"][3] > 1.0 for h in res["history"])   # clipping active
    assert_flat_parity(res)
    assert exact_fraction(res) > 0.99


def test_llama_like_zero2_rank0_periodic_overflow():
    """fp16 gradients ~N(0, 1e-4) x dynamic scale from 2^16, window 1000, rank 0
    of N=8 with shard-local gradients (after reduce-scatter), inf injected every
    50 steps, AdamW lr 1e-4 wd 0.1, 100 steps."""
    S = 262_147
    inj = {}
    for k, step in enumerate(range(50, 101, 50)):
        j = synth.seeded_indices(0x5EED0003, 200 + k, 1, 0, S)[0]
        inj[step] = [(0, j, INF16)]
    case = FlatCase(numel=8 * S, world=8, shards=(0,), shard_local_grads=True,
                    gdtype=O.FP16, lr=1e-4, wd=0.1, dynamic=True, init_scale=2.0 ** 16,
                    window=1000, sigma=1e-4, steps=100, seed=0x5EED0003, inject=inj)
    res = run_flat(case, check_every_step=False)
    sk = [h["step"] for h in res["history"] if h["gpu"][0]]
    assert sk == [50, 100]
    assert res["scaler"][0][0] == (2.0 ** 14, 0, 98, 2, 1)
    assert_flat_parity(res)


@pytest.mark.parametrize("stash", [True, False])
def test_fused_reduce_r8_k4_clip(stash):
    """8 simulated ranks x 4 micro-steps of fp16 shard gradients ~N(0, 1e-3) x
    1024, summed and divided by N*K = 32, AdamW lr 2e-4 wd 0.01, clip 1.0."""
    case = FlatCase(numel=300_007, world=1, ranks=8, micro=4, gdtype=O.FP16, lr=2e-4,
                    wd=0.01, max_norm=1.0, init_scale=1024.0, sigma=1e-3, steps=3,
                    divisor=32.0, seed=0x5EED0004, stash=stash, shard_local_grads=True)
    res = run_flat(case)
    assert_flat_parity(res)


def test_per_tensor_list_llama_shapes():
    """73 tensors with Llama-3-8B shapes (every dimension / 64): embedding plus
    8 decoder layers; bf16 gradients ~N(0, 1e-3), AdamW lr 1e-4 wd 0.1, clip 1.0."""
    shapes = llama_like_shapes(layers=8, div=64)
    assert len(shapes) == 73
    numels = [int(np.prod(s)) for s in shapes]
    res = run_list(numels, steps=3)
    assert_flat_parity(res)


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("n", [1, 7, 8, 9, 2047, 2048, 2049, 4099, 8 * 2048 * 4 + 5])
def test_sizes_around_the_tile(n):
    case = FlatCase(numel=n, gdtype=O.FP16, lr=1e-3, wd=0.01, max_norm=0.05,
                    init_scale=4.0, sigma=1e-2, steps=3)
    assert_flat_parity(run_flat(case))


@pytest.mark.parametrize("numel,world", [(3, 4), (1, 4), (5, 8), (0, 2)])
def test_all_padding_shards(numel, world):
    """Shards with no real element still take the global decision and advance
    their scaler; real shards match the oracle."""
    case = FlatCase(numel=numel, world=world, ranks=2, gdtype=O.FP16, dynamic=True,
                    init_scale=8.0, max_norm=0.5, steps=3)
    res = run_flat(case)
    assert_flat_parity(res)
    for r, (g, ref) in res["scaler"].items():
        assert g[2] == 3


@pytest.mark.parametrize("misalign", [1, 3])
def test_misaligned_buffers_take_the_element_path(misalign):
    case = FlatCase(numel=50_001, world=3, ranks=2, gdtype=O.BF16, lr=1e-3, wd=0.1,
                    max_norm=0.3, sigma=1e-2, steps=3, misalign=misalign)
    assert_flat_parity(run_flat(case))


def test_vector_and_element_paths_agree_bit_for_bit():
    base = dict(numel=40_000, world=1, ranks=3, gdtype=O.FP16, lr=1e-3, wd=0.01,
                init_scale=64.0, sigma=1e-2, steps=3)
    a = run_flat(FlatCase(misalign=0, **base))
    b = run_flat(FlatCase(misalign=1, **base))
    for x, y in zip(a["gpu"][0], b["gpu"][0]):
        assert (x.view(np.uint8) == y.view(np.uint8)).all()


@pytest.mark.parametrize("inject", [
    [(0, 1234, INF16)], [(1, 1234, NINF16)], [(0, 99_999, NAN16)],
    [(0, 5, INF16), (1, 5, NINF16)],
], ids=["+inf", "-inf", "nan", "+inf-inf"])
def test_overflow_kinds_skip(inject):
    case = FlatCase(numel=100_000, world=2, ranks=2, gdtype=O.FP16, dynamic=True,
                    init_scale=512.0, steps=3, inject={2: inject}, max_norm=1.0)
    res = run_flat(case)
    assert [h["gpu"][0] for h in res["history"]] == [0, 1, 0]
    assert_flat_parity(res)


def test_largest_fp16_values_do_not_overflow():
    inj = {1: [(b, j, 0x7BFF) for b in range(2) for j in range(0, 4096, 7)]}
    case = FlatCase(numel=10_000, ranks=2, gdtype=O.FP16, init_scale=1.0, steps=2,
                    inject=inj, max_norm=1.0)
    res = run_flat(case)
    assert res["history"][0]["gpu"][0] == 0
    assert_flat_parity(res)


@pytest.mark.parametrize("exp_bits", [0x5C00, 0x1F00], ids=["2^57", "2^-65"])
def test_extreme_bf16_magnitudes_in_the_norm(exp_bits):
    """Gradients near 2^57 (squares near the binary32 overflow range) and near
    2^-65 (squares below binary32's normal range) still give the oracle's norm."""
    inj = {s: [(0, j, exp_bits | (j & 0x7F)) for j in range(0, 3000, 3)] for s in (1, 2)}
    case = FlatCase(numel=6000, gdtype=O.BF16, steps=2, max_norm=1.0, sigma=1e-30,
                    inject=inj)
    res = run_flat(case)
    assert_flat_parity(res)


def test_stash_and_reread_agree_bit_for_bit():
    base = dict(numel=70_001, world=1, ranks=4, micro=2, gdtype=O.FP16, lr=1e-3,
                max_norm=0.5, init_scale=32.0, steps=3, shard_local_grads=True)
    a = run_flat(FlatCase(stash=True, **base))
    b = run_flat(FlatCase(stash=False, **base))
    for x, y in zip(a["gpu"][0], b["gpu"][0]):
        assert (x.view(np.uint8) == y.view(np.uint8)).all()


def test_runs_are_deterministic():
    case = FlatCase(numel=300_000, world=2, ranks=2, gdtype=O.BF16, max_norm=0.1,
                    sigma=1e-2, steps=3)
    a = run_flat(case)
    b = run_flat(case)
    assert [h["gpu"] for h in a["history"]] == [h["gpu"] for h in b["history"]]
    for r in a["gpu"]:
        for x, y in zip(a["gpu"][r], b["gpu"][r]):
            assert (x.view(np.uint8) == y.view(np.uint8)).all()


def test_resume_is_bit_exact():
    """Ten steps straight equal five steps, a save of (master, m, v, scaler) and
    a restore into a fresh handle, then five more steps."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n = 50_000
    cfg = z.make_config(numel=n, world=1, grad_dtype=z.FP16, lr=1e-3, weight_decay=0.01,
                        max_grad_norm=0.5, dynamic_scale=True, init_scale=256.0,
                        scale_window=3)
    p0 = torch.from_numpy(synth.normal_np(5, 0, 0, n, 0.02, synth.F32)).to(dev)
    grads = [synth.normal_torch(5, 1, n, 0.5, synth.F16, device=dev, offset=s * n)
             for s in range(10)]
    grads[6][17] = float("inf")

    def fresh():
        return [p0.clone(), torch.zeros(n, device=dev), torch.zeros(n, device=dev),
                torch.zeros(n, dtype=torch.float16, device=dev)]

    def steps(h, st, lo, hi):
        for s in range(lo, hi):
            z.zero_opt_step(h, 0, z.make_buffers(*st, [grads[s]]))

    h1 = z.zero_opt_create(cfg)
    a = fresh()
    steps(h1, a, 0, 10)
    h2 = z.zero_opt_create(cfg)
    b = fresh()
    steps(h2, b, 0, 5)
    saved = [x.clone() for x in b]
    sc = z.zero_opt_loss_scale(h2, 0)
    z.zero_opt_destroy(h2)
    h3 = z.zero_opt_create(cfg)
    z.zero_opt_set_loss_scale(h3, 0, sc)
    steps(h3, saved, 5, 10)
    torch.cuda.synchronize()
    for x, y in zip(a, saved):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    assert z.zero_opt_loss_scale(h1, 0).as_tuple() == z.zero_opt_loss_scale(h3, 0).as_tuple()
    z.zero_opt_destroy(h1)
    z.zero_opt_destroy(h3)


def test_local_step_equals_stats_fold_step():
    """For one shard that is the whole world, the asynchronous local step and
    the statistics -> fold -> step sequence agree bit for bit."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n = 123_457
    cfg = z.make_config(numel=n, world=1, grad_dtype=z.BF16, lr=1e-3, max_grad_norm=0.2,
                        dynamic_scale=False, init_scale=1.0)
    g = synth.normal_torch(3, 1, n, 1e-2, synth.BF16, device=dev)
    p0 = torch.from_numpy(synth.normal_np(3, 0, 0, n, 0.02, synth.F32)).to(dev)
    out = []
    for use_fold in (False, True):
        h = z.zero_opt_create(cfg)
        st = [p0.clone(), torch.zeros(n, device=dev), torch.zeros(n, device=dev),
              torch.zeros(n, dtype=torch.bfloat16, device=dev)]
        b = z.make_buffers(*st, [g])
        for _ in range(3):
            if use_fold:
                G = z.zero_opt_fold_stats([z.zero_opt_grad_stats(h, 0, b)])
                z.zero_opt_step(h, 0, b, global_stats=G)
            else:
                z.zero_opt_step(h, 0, b)
        torch.cuda.synchronize()
        out.append(st)
        z.zero_opt_destroy(h)
    for x, y in zip(*out):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


def test_cast_matches_cuda_intrinsics_sample():
    """The oracle's RNE casts equal CUDA's conversion on a sample of values,
    through the 16-bit copy the step writes (lr = 0 keeps master = input)."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 32, 1 << 16, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = np.where(np.isfinite(x) & (np.abs(x) < 6e4), x, 1.0).astype(np.float32)
    n = x.size
    for dt, code in ((torch.float16, z.FP16), (torch.bfloat16, z.BF16)):
        cfg = z.make_config(numel=n, world=1, grad_dtype=code, lr=0.0, weight_decay=0.0,
                            dynamic_scale=False, init_scale=1.0)
        h = z.zero_opt_create(cfg)
        st = [torch.from_numpy(x.copy()).to(dev), torch.zeros(n, device=dev),
              torch.zeros(n, device=dev), torch.zeros(n, dtype=dt, device=dev)]
        z.zero_opt_step(h, 0, z.make_buffers(*st, [torch.zeros(n, dtype=dt, device=dev)]))
        torch.cuda.synchronize()
        got = st[3].cpu().view(torch.int16).numpy().view(np.uint16)
        ref = O.f32_to_16(x, O.FP16 if code == z.FP16 else O.BF16)
        assert (got == ref).all()
        z.zero_opt_destroy(h)


def test_hysteresis_and_warmup_lr():
    """Hysteresis 2 (the scale falls on every second overflow) with a WarmupLR
    schedule (linear over 6 updates) and clipping, 14 steps with overflows on
    steps 3, 4, 7 and 11; every step's scaler state matches the oracle."""
    inj = {s: [(0, 1000 + s, INF16)] for s in (3, 4, 7, 11)}
    case = FlatCase(numel=200_003, world=2, ranks=2, gdtype=O.FP16, lr=1e-3, wd=0.01,
                    max_norm=0.5, dynamic=True, init_scale=256.0, window=3, hysteresis=2,
                    warmup=(1e-4, 2e-3, 6), sigma=1e-3, steps=14, inject=inj)
    res = run_flat(case)
    assert [h["gpu"][0] for h in res["history"]] == [int(s in inj) for s in range(1, 15)]
    assert_flat_parity(res)


@pytest.mark.parametrize("gdtype", [O.BF16, O.FP16])
def test_low_precision_master(gdtype):
    """master16: no fp32 master array, the 16-bit parameters are the masters
    (widened, updated, stored back rounded).  Two shards, clipping, weight
    decay, dynamic scale with an overflow on step 3; the 16-bit masters must
    match the oracle's within one ulp and m, v within the state tolerance."""
    inj = {3: [(1, 777, INF16 if gdtype == O.FP16 else 0x7F80)]}
    case = FlatCase(numel=300_007, world=2, ranks=2, gdtype=gdtype, lr=1e-3, wd=0.01,
                    max_norm=0.5, dynamic=True, init_scale=16.0, sigma=1e-2, steps=5,
                    inject=inj, master16=True)
    res = run_flat(case)
    assert [h["gpu"][0] for h in res["history"]] == [0, 0, 1, 0, 0]
    assert_flat_parity(res)
    # the 16-bit masters agree bit for bit on at least 99.9% of the elements
    same = tot = 0
    for r in res["gpu"]:
        g16 = res["gpu"][r][0].view(np.uint32)
        o16 = res["ref"][r][0].view(np.uint32)
        same += int((g16 == o16).sum())
        tot += g16.size
    assert same >= 0.999 * tot, same / tot


@pytest.mark.parametrize("stash", [True, False])
def test_low_precision_master_tensor_list(stash):
    """master16 on a per-tensor list with R*K = 2*3 fp16 buffers (the
    multi-buffer pass 1, and the stash when asked), ragged tensor sizes."""
    res = run_list([5000, 2049, 1, 70_001, 4096], gdtype=O.FP16, lr=1e-3, wd=0.01,
                   max_norm=0.5, sigma=1e-3, steps=3, ranks=2, micro=3, stash=stash,
                   master16=True)
    assert_flat_parity(res)


def test_device_folded_statistics_equal_the_host_fold():
    """zero_opt_grad_stats_async + zero_opt_step_folded (statistics kept and
    folded on the device) against zero_opt_grad_stats + zero_opt_fold_stats +
    zero_opt_step: three ranks of one buffer, four steps with an overflow on
    the third, bit-identical states, decisions and scaler states."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    numel, world, R = 90_001, 3, 2
    cfg = z.make_config(numel=numel, world=world, grad_dtype=z.BF16, lr=1e-3,
                        weight_decay=0.01, max_grad_norm=0.3, dynamic_scale=True,
                        init_scale=32.0)
    hs = [z.zero_opt_create(cfg) for _ in range(2)]
    _, _, S, P = z.zero_opt_shard_bounds(hs[0], 0)
    p0 = torch.from_numpy(synth.normal_np(0x5EED0601, 0, 0, P, 0.02, synth.F32)).to(dev)
    states = [[[p0[r * S:(r + 1) * S].clone(), torch.zeros(S, device=dev),
                torch.zeros(S, device=dev)] for r in range(world)] for _ in range(2)]
    p16 = [torch.zeros(P, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    stats = torch.zeros(16 * world, dtype=torch.uint8, device=dev)
    for step in range(1, 5):
        grads = [synth.normal_torch(0x5EED0601, 1 + b, P, 1e-2 * 32.0, synth.BF16, device=dev,
                                    offset=step * P) for b in range(R)]
        if step == 3:
            grads[1][numel - 5] = float("inf")
        # device fold
        bufs = [z.make_buffers(*states[0][r], p16[0], grads) for r in range(world)]
        for r in range(world):
            z.zero_opt_grad_stats_async(hs[0], r, bufs[r], stats[16 * r:16 * (r + 1)])
        for r in range(world):
            z.zero_opt_step_folded(hs[0], r, bufs[r], stats, world)
        dec = z.zero_opt_last_step(hs[0])
        # host fold
        bufs2 = [z.make_buffers(*states[1][r], p16[1], grads) for r in range(world)]
        G = z.zero_opt_fold_stats([z.zero_opt_grad_stats(hs[1], r, bufs2[r])
                                   for r in range(world)])
        for r in range(world):
            z.zero_opt_step(hs[1], r, bufs2[r], global_stats=G)
        ref = z.zero_opt_last_step(hs[1])
        assert (dec.skipped, dec.sumsq, dec.coef, dec.t) == (ref.skipped, ref.sumsq, ref.coef,
                                                             ref.t) or (dec.skipped == ref.skipped == 1)
        assert dec.skipped == (1 if step == 3 else 0)
        for r in range(world):
            assert z.zero_opt_loss_scale(hs[0], r).as_tuple() == \
                z.zero_opt_loss_scale(hs[1], r).as_tuple()
    torch.cuda.synchronize()
    for r in range(world):
        for a, b in zip(states[0][r], states[1][r]):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(p16[0].view(torch.int16), p16[1].view(torch.int16))
    for h in hs:
        z.zero_opt_destroy(h)


@pytest.mark.parametrize("t0,warmup", [(65_533, (0.0, 0.0, 0)), (65_534, (1e-5, 1e-3, 70_000))])
def test_steps_across_the_bias_correction_table(t0, warmup):
    """The bias corrections of steps 1..65536 come from a per-handle table, later
    ones from pow on the device: steps t0+1 .. t0+4 straddle the boundary
    (with WarmupLR still ramping in the second case) and must match the
    oracle bit for bit, as the scaler counters must."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n = 50_003
    cfg = z.make_config(numel=n, world=1, grad_dtype=z.BF16, lr=1e-3, weight_decay=0.01,
                        dynamic_scale=False, init_scale=1.0, warmup=warmup)
    h = z.zero_opt_create(cfg)
    st = z.zero_opt_loss_scale(h, 0)
    st.t = t0
    z.zero_opt_set_loss_scale(h, 0, st)
    hp = O.hparams(lr=1e-3, weight_decay=0.01, warmup=warmup)
    sc = O.scaler(1.0)
    sc.t = t0
    orc = O.default()
    p0 = synth.normal_np(0x5EED0701, 0, 0, n, 0.02, synth.F32)
    state = [torch.from_numpy(p0).to(dev), torch.zeros(n, device=dev), torch.zeros(n, device=dev),
             torch.zeros(n, dtype=torch.bfloat16, device=dev)]
    ref = [p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    for step in range(1, 5):
        g = synth.normal_np(0x5EED0701, 1, step * n, n, 1e-2, synth.BF16)
        gt = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).to(dev)
        z.zero_opt_step(h, 0, z.make_buffers(*state, [gt]))
        orc.step(hp, sc, [g], O.BF16, *ref, O.BF16, 1.0)
        assert z.zero_opt_loss_scale(h, 0).as_tuple() == sc.as_tuple()
    torch.cuda.synchronize()
    assert sc.t == t0 + 4
    for a, b in zip(state[:3], ref[:3]):
        assert (a.cpu().numpy().view(np.uint32) == b.view(np.uint32)).all()
    assert (to_np16(state[3]) == ref[3]).all()
    z.zero_opt_destroy(h)


@pytest.mark.parametrize("ranks", [1, 2], ids=["one-buffer", "two-buffers"])
@pytest.mark.parametrize("master16", [False, True], ids=["fp32-masters", "16-bit-masters"])
@pytest.mark.parametrize("g,p", [(O.FP16, O.BF16), (O.BF16, O.FP16)],
                         ids=["fp16-grads-bf16-params", "bf16-grads-fp16-params"])
def test_mixed_16bit_types(g, p, master16, ranks):
    """Gradients in one 16-bit type and parameters in the other (param_dtype),
    with fp32 or 16-bit masters, over two shards with folded statistics,
    dynamic scaling and clipping."""
    case = FlatCase(numel=300_007, world=2, ranks=ranks, gdtype=g, pdtype=p, lr=1e-3, wd=0.01,
                    max_norm=0.5, dynamic=True, init_scale=256.0, window=3, sigma=1e-3,
                    steps=5, master16=master16, seed=0x5EED0D00)
    res = run_flat(case)
    assert_flat_parity(res)


@pytest.mark.parametrize("master16", [False, True], ids=["fp32-masters", "16-bit-masters"])
def test_list_with_mixed_16bit_types(master16):
    """The per-tensor list with bf16 gradients and fp16 parameters: ragged
    tensor sizes, two gradient buffers (the multi-buffer pass 1)."""
    res = run_list([5000, 2049, 1, 70_001, 4096], gdtype=O.BF16, pdtype=O.FP16, lr=1e-3,
                   wd=0.01, max_norm=0.5, steps=3, ranks=2, master16=master16)
    assert_flat_parity(res)


@pytest.mark.parametrize("master16", [False, True], ids=["fp32-masters", "16-bit-masters"])
def test_state_alignment_selects_the_access_width_not_the_result(master16):
    """Pass 2 moves the fp32 state with 256-bit accesses when master, m and v
    are 32-byte aligned and with 128-bit ones when they are only 16-byte
    aligned.  The same three steps on both layouts give bit-identical state."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n = 300_007
    cfg = z.make_config(numel=n, world=1, grad_dtype=z.BF16, lr=1e-3, weight_decay=0.01,
                        max_grad_norm=0.5, dynamic_scale=False, init_scale=1.0,
                        master16=master16)
    p0 = synth.normal_np(0x5EED0E00, 0, 0, n, 0.02, synth.F32)
    q0 = O.f32_to_16(p0, O.BF16)
    grads = [synth.normal_torch(0x5EED0E00, 1, n, 1e-2, synth.BF16, device=dev, offset=s * n)
             for s in range(3)]

    def run(shift):
        # fp32 arrays at `shift` floats past a 512-byte aligned allocation
        arrs = [torch.zeros(n + 8, device=dev)[shift:shift + n] for _ in range(3)]
        arrs[0].copy_(torch.from_numpy(p0))
        p16 = torch.from_numpy(q0.view(np.int16).copy()).view(torch.bfloat16).to(dev)
        h = z.zero_opt_create(cfg)
        for g in grads:
            z.zero_opt_step(h, 0, z.make_buffers(None if master16 else arrs[0], arrs[1],
                                                 arrs[2], p16, [g]))
        torch.cuda.synchronize()
        z.zero_opt_destroy(h)
        return [a.clone() for a in arrs], p16.clone()

    (a, ap), (b, bp) = run(0), run(4)
    assert arrs_equal(a, b, master16)
    assert torch.equal(ap.view(torch.int16), bp.view(torch.int16))


def test_stash_alignment_selects_the_load_width_not_the_result():
    """Pass 2 reads the binary32 stash with one 256-bit load per lane when the
    stash is 32-byte aligned and with two 128-bit loads when it is only
    16-byte aligned.  Three steps of six gradient buffers through the stash,
    on both layouts, give bit-identical state, and both match the oracle."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n, R, K = 200_003, 3, 2
    cfg = z.make_config(numel=n, world=1, grad_dtype=z.FP16, lr=1e-3, weight_decay=0.01,
                        max_grad_norm=0.5, dynamic_scale=False, init_scale=1.0)
    p0 = synth.normal_np(0x5EED0E10, 0, 0, n, 0.02, synth.F32)
    steps = [[synth.normal_torch(0x5EED0E10, 1 + s * R * K + b, n, 1e-3, synth.F16, device=dev)
              for b in range(R * K)] for s in range(3)]

    def run(shift):
        master = torch.from_numpy(p0.copy()).to(dev)
        m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
        p16 = torch.zeros(n, dtype=torch.float16, device=dev)
        # the stash `shift` floats past a 512-byte aligned allocation
        stash = torch.zeros(n + 8, device=dev)[shift:shift + n]
        h = z.zero_opt_create(cfg)
        for g in steps:
            z.zero_opt_step(h, 0, z.make_buffers(master, m, v, p16, g, n_ranks=R, n_micro=K,
                                                 grads_shard_local=True, stash=stash))
        torch.cuda.synchronize()
        z.zero_opt_destroy(h)
        return [master, m, v], p16

    (a, ap), (b, bp) = run(0), run(4)
    assert arrs_equal(a, b, False)
    assert torch.equal(ap.view(torch.int16), bp.view(torch.int16))
    orc = O.default()
    hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=0.5, dynamic_scale=False)
    sc = O.scaler(1.0)
    ref = (p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16))
    for g in steps:
        orc.step(hp, sc, [to_np16(x) for x in g], O.FP16, *ref, O.FP16, float(R * K))
    assert_state("master", a[0].cpu().numpy(), ref[0])
    assert_state("m", a[1].cpu().numpy(), ref[1])
    assert_state("v", a[2].cpu().numpy(), ref[2])
    assert ulp16_diff(to_np16(ap), ref[3]) <= 1


@pytest.mark.parametrize("stash", [False, True], ids=["reread", "stash"])
def test_buffer_limit_of_1024_matches_the_oracle_and_1025_is_refused(stash):
    """R*K = 32 x 32 = 1024 gradient buffers, the most one step takes, over a
    ragged shard of 3001 elements: three clipped steps match the oracle, with
    the sums re-read in pass 2 and through the stash.  41 x 25 = 1025 buffers
    are refused with ZERO_EINVAL before anything is launched."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    n, R, K = 3001, 32, 32
    cfg = z.make_config(numel=n, world=1, grad_dtype=z.FP16, lr=1e-3, weight_decay=0.01,
                        max_grad_norm=0.5, dynamic_scale=False, init_scale=1.0)
    p0 = synth.normal_np(0x5EED0E20, 0, 0, n, 0.02, synth.F32)
    master = torch.from_numpy(p0.copy()).to(dev)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    p16 = torch.zeros(n, dtype=torch.float16, device=dev)
    st = torch.zeros(n, device=dev) if stash else None
    h = z.zero_opt_create(cfg)
    orc = O.default()
    hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=0.5, dynamic_scale=False)
    sc = O.scaler(1.0)
    ref = (p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16))
    try:
        for step in range(3):
            g = [synth.normal_torch(0x5EED0E20, 1 + step * R * K + b, n, 1e-3, synth.F16,
                                    device=dev) for b in range(R * K)]
            z.zero_opt_step(h, 0, z.make_buffers(master, m, v, p16, g, n_ranks=R, n_micro=K,
                                                 grads_shard_local=True, stash=st))
            orc.step(hp, sc, [to_np16(x) for x in g], O.FP16, *ref, O.FP16, float(R * K))
        torch.cuda.synchronize()
        assert_state("master", master.cpu().numpy(), ref[0])
        assert_state("m", m.cpu().numpy(), ref[1])
        assert_state("v", v.cpu().numpy(), ref[2])
        assert ulp16_diff(to_np16(p16), ref[3]) <= 1
        launched = z.zero_opt_launch_count(h)
        g = [torch.zeros(n, dtype=torch.float16, device=dev)] * (41 * 25)
        with pytest.raises(z.ZeroOptError) as e:
            z.zero_opt_step(h, 0, z.make_buffers(master, m, v, p16, g, n_ranks=41, n_micro=25,
                                                 grads_shard_local=True, stash=st))
        assert e.value.status == z.ZERO_EINVAL
        assert z.zero_opt_launch_count(h) == launched
    finally:
        z.zero_opt_destroy(h)


def arrs_equal(a, b, master16):
    import torch
    first = 1 if master16 else 0         # the master array is unused with 16-bit masters
    return all(torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(a[first:], b[first:]))
