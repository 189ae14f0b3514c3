"""Pins of the parity oracle against what the pages and mathematics fix.

Every function takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a value printed by the pages, a closed form, an
invariant, a library routine or brute force.  ``test_oracle_pins`` runs them
on the real oracle; ``test_oracle_mutants`` runs them on copies of the oracle
with one planted mistake each and requires that some pin fails.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import oracle as O
import synth
from conftest import read_golden

F16, BF16 = O.FP16, O.BF16


def _h(vals, dtype=F16):
    """Exact 16-bit bit patterns of small decimal values (via numpy/torch)."""
    x = np.asarray(vals, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16).copy()
    import torch
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _f(bits, dtype=F16):
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    import torch
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def _state(n, p0=None):
    master = np.zeros(n, np.float32) if p0 is None else np.asarray(p0, np.float32).copy()
    return master, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)


def _close(a, b, rel, abs_=0.0):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    ok = np.abs(a - b) <= np.maximum(rel * np.abs(b), abs_)
    assert ok.all(), f"max diff {np.max(np.abs(a - b))} at {np.argmax(~ok)}: {a[~ok][:4]} vs {b[~ok][:4]}"


# ---------------------------------------------------------------- a0 and forms

def pin_shard_bounds_bruteforce(orc):
    """Every element of the padded buffer lies in exactly one shard; shards are
    equal, padding is shorter than N and only the last shards hold it
    ("ZeRO三阶段": cut into N parts by GPU count)."""
    for numel in range(0, 41):
        for world in range(1, 10):
            owner = np.full(max(numel, 1), -1)
            lens = set()
            for r in range(world):
                b, e, s, p = orc.shard_bounds(numel, world, r)
                lens.add(s)
                assert p == s * world and p >= numel and p - numel < world
                assert b == r * s and b <= e <= b + s and e <= max(numel, b)
                for j in range(b, e):
                    assert owner[j] == -1
                    owner[j] = r
            assert len(lens) == 1
            assert numel == 0 or (owner[:numel] >= 0).all()


def pin_shard_bounds_workloads(orc):
    # 1,000,003 parameters over 4 ranks pad to 1,000,004: shards of 250,001,
    # the last one with 250,000 real elements and one padding element.
    assert orc.shard_bounds(1_000_003, 4, 3) == (750_003, 1_000_003, 250_001, 1_000_004)
    assert orc.shard_bounds(1_000_003, 4, 0) == (0, 250_001, 250_001, 1_000_004)
    # 8,030,261,248 over 8 ranks divides exactly.
    assert orc.shard_bounds(8_030_261_248, 8, 0) == (0, 1_003_782_656, 1_003_782_656, 8_030_261_248)
    assert orc.shard_bounds(8_030_261_248, 8, 7)[1] == 8_030_261_248
    # fewer elements than ranks: trailing shards are all padding
    assert orc.shard_bounds(3, 4, 3) == (3, 3, 1, 4)
    assert orc.shard_bounds(1, 4, 2) == (2, 2, 1, 4)


def pin_memory_forms(orc):
    """[JWZ] §1.2: M_DDP = 16Ψ; M_ZeRO-1 = 4Ψ + 12Ψ/N; M_ZeRO-2 = 2Ψ + 14Ψ/N;
    M_ZeRO-3 = 16Ψ/N, exact when N divides Ψ; [CSDN] §2.1: 7B -> 112 GB."""
    for numel, world, stage, expect in read_golden("memory_7b.txt"):
        assert orc.memory_bytes(int(numel), int(world), int(stage)) == int(expect)
    for psi, n in [(8_030_261_248, 8), (124_439_808, 1), (1_000_004, 4), (4096, 64),
                   (2_270_232_576, 2), (600, 3)]:
        P = Fraction(psi)
        forms = [16 * P, 4 * P + 12 * P / n, 2 * P + 14 * P / n, 16 * P / n]
        for stage, f in enumerate(forms):
            assert f.denominator == 1
            assert orc.memory_bytes(psi, n, stage) == int(f), (psi, n, stage)
    # ZeRO on one rank is plain data parallelism.
    for stage in range(4):
        assert orc.memory_bytes(1_000_003, 1, stage) == 16 * 1_000_003
    # [AIDH]: stage 1 saves about 4x and stage 2 about 8x; those are the limits
    # of 16/(4 + 12/N) and 16/(2 + 14/N) for large N.
    psi, n = 10 ** 12, 10 ** 6
    assert abs(16 * psi / orc.memory_bytes(psi, n, 1) - 4) < 1e-4
    assert abs(16 * psi / orc.memory_bytes(psi, n, 2) - 8) < 1e-4
    # Llama-3-8B sizes over 8 ranks (the closed forms as integers).
    assert orc.memory_bytes(8_030_261_248, 8, 0) == 128_484_179_968
    assert orc.memory_bytes(8_030_261_248, 8, 1) == 44_166_436_864
    assert orc.memory_bytes(8_030_261_248, 8, 2) == 30_113_479_680
    assert orc.memory_bytes(8_030_261_248, 8, 3) == 16_060_522_496
    assert orc.memory_bytes(5, 0, 0) == -1 and orc.memory_bytes(5, 1, 4) == -1


# ---------------------------------------------------------------- casts

def _structured_patterns(hi_bits, lo_bits, seed):
    rng = np.random.default_rng(seed)
    lo_mask = (1 << lo_bits) - 1
    half = 1 << (lo_bits - 1)
    lows = [0, 1, half - 1, half, half + 1, lo_mask] + list(rng.integers(0, lo_mask, 10))
    hi = np.arange(0, 1 << hi_bits, dtype=np.uint64) << np.uint64(lo_bits)
    pats = [(hi | np.uint64(lo)).astype(np.uint32) for lo in lows]
    pats.append(rng.integers(0, 1 << 32, 1 << 20, dtype=np.uint64).astype(np.uint32))
    return np.concatenate(pats)


def pin_cast_fp16_vs_numpy(orc):
    """Round-to-nearest-even binary32 -> binary16 against numpy's conversion,
    on every sign/exponent/10-bit-mantissa prefix with the tie, near-tie and
    random low bits, plus random patterns; decode of all 65536 codes."""
    bits = _structured_patterns(19, 13, 1)
    x = bits.view(np.float32)
    ours = orc.f32_to_16(x, F16)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert (ours[~nan] == ref[~nan]).all(), np.flatnonzero(ours[~nan] != ref[~nan])[:5]
    assert np.isnan(ours[nan].view(np.float16)).all()
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = orc.f16_to_f32(codes, F16)
    ref = codes.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert (dec[~nan].view(np.uint32) == ref[~nan].view(np.uint32)).all()
    assert np.isnan(dec[nan]).all()


def pin_cast_bf16_vs_torch(orc):
    import torch
    bits = _structured_patterns(16, 16, 2)
    x = bits.view(np.float32)
    ours = orc.f32_to_16(x, BF16)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert (ours[~nan] == ref[~nan]).all(), np.flatnonzero(ours[~nan] != ref[~nan])[:5]
    assert np.isnan(_f(ours[nan], BF16)).all()
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = orc.f16_to_f32(codes, BF16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert (dec[~nan].view(np.uint32) == ref[~nan].view(np.uint32)).all()


# ---------------------------------------------------------------- Adam closed forms

_G8 = [1.0, -2.0, 0.5, -0.25, 3.0, 24.0, -7e-3, 0.0]


def pin_first_step_bias_corrected(orc):
    """With bias correction the first update is -lr * g / (|g| + eps) for any
    beta: m_hat = g and v_hat = g^2 after one step; m = (1-b1) g, v = (1-b2) g^2
    pin the unscale g = s / (scale * D)."""
    scale, D, lr = 2048.0, 4.0, 1e-3
    hp = O.hparams(lr=lr, betas=(0.9, 0.999), eps=1e-8, dynamic_scale=True)
    st = O.scaler(scale)
    # four ranks' buffers; their sum is 4 * scale * x for x in _G8
    x = np.asarray(_G8, np.float64)
    bufs = [_h(x * scale) for _ in range(4)]
    s_exact = 4 * _f(bufs[0])
    g = s_exact / (scale * D)
    master, m, v, p16 = _state(8)
    orc.step(hp, st, bufs, F16, master, m, v, p16, F16, D)
    _close(m, 0.1 * g, 2e-7)
    _close(v, 0.001 * g * g, 5e-7)
    _close(master, -lr * g / (np.abs(g) + 1e-8), 2e-6)
    assert st.t == 1 and not st.last_skipped
    # the 16-bit copy is the rounding of the master copy
    assert (p16 == _h(master)).all()


def pin_constant_grad_bias_corrected(orc):
    """Constant g: m_t = (1-b1^t) g and v_t = (1-b2^t) g^2, so every bias-
    corrected step moves the parameter by -lr g / (|g| + eps)."""
    lr = 2e-3
    hp = O.hparams(lr=lr, betas=(0.8, 0.95), eps=1e-8)
    st = O.scaler(1.0)
    bufs = [_h(_G8)]
    g = _f(bufs[0])
    master, m, v, p16 = _state(8)
    prev = master.astype(np.float64)
    for t in range(1, 7):
        orc.step(hp, st, bufs, F16, master, m, v, p16, F16, 1.0)
        _close(m, (1 - 0.8 ** t) * g, 1e-6)
        _close(v, (1 - 0.95 ** t) * g * g, 2e-6)
        _close(master - prev, -lr * g / (np.abs(g) + 1e-8), 1e-5, 1e-12)
        prev = master.astype(np.float64)
    assert st.t == 6


def pin_constant_grad_no_bias_correction(orc):
    """Without bias correction (the "Python 演示" Adam) a constant g moves the
    parameter by -lr (1-b1^t) g / (sqrt(1-b2^t) |g| + eps) at step t."""
    lr = 1e-2
    hp = O.hparams(lr=lr, betas=(0.9, 0.99), eps=1e-8, bias_correction=False)
    st = O.scaler(1.0)
    bufs = [_h(_G8)]
    g = _f(bufs[0])
    master, m, v, p16 = _state(8)
    prev = master.astype(np.float64)
    for t in range(1, 6):
        orc.step(hp, st, bufs, F16, master, m, v, p16, F16, 1.0)
        expect = -lr * (1 - 0.9 ** t) * g / (math.sqrt(1 - 0.99 ** t) * np.abs(g) + 1e-8)
        _close(master - prev, expect, 1e-5, 1e-12)
        prev = master.astype(np.float64)


def pin_aiqz_demo(orc):
    """The demo's first step: all-ones gradient divided by world 4, Adam
    without bias correction, eps in the denominator."""
    kv = {k: float(v) for k, v in read_golden("aiqz_demo.txt")}
    hp = O.hparams(lr=kv["lr"], betas=(kv["beta1"], kv["beta2"]), eps=kv["eps"],
                   bias_correction=False)
    st = O.scaler(1.0)
    n = 1024
    bufs = [_h(np.full(n, kv["grad"]))]
    master, m, v, p16 = _state(n)
    orc.step(hp, st, bufs, F16, master, m, v, p16, F16, kv["world"])
    _close(master, np.full(n, kv["delta"]), 1e-6)
    _close(m, np.full(n, 0.1 * 0.25), 1e-7)
    _close(v, np.full(n, 0.001 * 0.0625), 1e-6)


def pin_lr_zero(orc):
    """lr = 0 leaves the master weights bit-identical while m and v move."""
    hp = O.hparams(lr=0.0, betas=(0.9, 0.999), weight_decay=0.1)
    st = O.scaler(1.0)
    bufs = [_h(_G8)]
    g = _f(bufs[0])
    p0 = np.linspace(-1, 1, 8).astype(np.float32)
    master, m, v, p16 = _state(8, p0)
    orc.step(hp, st, bufs, F16, master, m, v, p16, F16, 1.0)
    assert (master.view(np.uint32) == p0.view(np.uint32)).all()
    _close(m, 0.1 * g, 2e-7)
    _close(v, 0.001 * g * g, 5e-7)


def pin_zero_betas(orc):
    """beta1 = beta2 = 0: no memory, m = g, v = g^2 and each step moves by
    -lr g / (|g| + eps) whatever the previous gradients were."""
    lr = 1e-3
    hp = O.hparams(lr=lr, betas=(0.0, 0.0))
    st = O.scaler(1.0)
    master, m, v, p16 = _state(8)
    rng = np.random.default_rng(5)
    for t in range(4):
        bufs = [_h(rng.normal(size=8) * 4)]
        g = _f(bufs[0])
        prev = master.astype(np.float64)
        orc.step(hp, st, bufs, F16, master, m, v, p16, F16, 1.0)
        _close(m, g, 0)
        _close(v, g * g, 1e-7)
        _close(master - prev, -lr * g / (np.abs(g) + 1e-8), 1e-5, 1e-12)


def pin_weight_decay_only(orc):
    """Zero gradients: AdamW only decays, p_k = p_0 (1 - lr wd)^k ([CSDN] §3.2
    AdamW with weight_decay)."""
    lr, wd = 0.01, 0.5
    hp = O.hparams(lr=lr, weight_decay=wd)
    st = O.scaler(1.0)
    p0 = np.linspace(-0.5, 0.5, 8).astype(np.float32)
    master, m, v, p16 = _state(8, p0)
    bufs = [np.zeros(8, np.uint16)]
    for k in range(1, 11):
        orc.step(hp, st, bufs, F16, master, m, v, p16, F16, 1.0)
        _close(master, p0.astype(np.float64) * (1 - lr * wd) ** k, 1e-6)
    assert (m == 0).all() and (v == 0).all()


def _textbook_adamw(p, m, v, s, scale, D, t, lr, b1, b2, eps, wd, max_norm):
    """Binary64 AdamW in the textbook form m_hat = m/(1-b1^t), v_hat = v/(1-b2^t),
    weight decay p <- p (1 - lr wd) before the Adam term."""
    g = s / (scale * D)
    if max_norm > 0:
        norm = np.sqrt(np.sum(g * g))
        g = g * min(1.0, max_norm / (norm + 1e-6))
    p = p * (1 - lr * wd)
    m = b1 * m + (1 - b1) * g
    v = b2 * v + (1 - b2) * g * g
    mh = m / (1 - b1 ** t)
    vh = v / (1 - b2 ** t)
    return p - lr * mh / (np.sqrt(vh) + eps), m, v


def pin_textbook_adamw_fp64(orc):
    """Several steps with loss scale, divisor, clipping and weight decay agree
    with binary64 textbook AdamW to within the binary32 rounding."""
    for lr, wd, max_norm in [(1e-3, 0.01, 0.5), (0.05, 2.0, 0.0), (3e-4, 0.1, 1e9)]:
        n, R, scale, steps = 64, 3, 512.0, 5
        b1, b2, eps = 0.9, 0.999, 1e-8
        hp = O.hparams(lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
                       max_grad_norm=max_norm)
        st = O.scaler(scale)
        p0 = synth.normal_np(11, 0, 0, n, 0.02, synth.F32)
        master, m, v, p16 = _state(n, p0)
        P, M, V = p0.astype(np.float64), np.zeros(n), np.zeros(n)
        for t in range(1, steps + 1):
            bufs = [synth.normal_np(11, 10 * t + r, 0, n, 1e-3 * scale, synth.F16) for r in range(R)]
            s = sum(_f(b) for b in bufs)   # exact in binary64
            orc.step(hp, st, bufs, F16, master, m, v, p16, F16, float(R))
            P, M, V = _textbook_adamw(P, M, V, s, scale, R, t, lr, b1, b2, eps, wd, max_norm)
            _close(master, P, 1e-5, 1e-9)
            _close(m, M, 1e-5, 1e-12)
            _close(v, V, 1e-5, 1e-16)


# ---------------------------------------------------------------- norm and clip

def pin_norm_vs_numpy(orc):
    """The reported norm is the L2 norm of the unscaled reduced gradient."""
    n, scale, D = 1000, 1024.0, 2.0
    bufs = [synth.normal_np(3, r, 0, n, 1e-3 * scale, synth.F16) for r in range(2)]
    s = orc.reduce(bufs, F16)
    assert (s == (_f(bufs[0]) + _f(bufs[1])).astype(np.float32)).all()
    st_ = orc.stats_of(s)
    assert abs(st_.sumsq - np.dot(s.astype(np.float64), s.astype(np.float64))) <= 1e-12 * st_.sumsq
    hp = O.hparams(max_grad_norm=0.0)
    d = orc.decide(hp, O.scaler(scale), st_, D)
    ref = np.linalg.norm(s.astype(np.float64)) / (scale * D)
    assert abs(d.norm - ref) <= 1e-12 * ref


def pin_clip_closed_form(orc):
    """16 equal gradients c = 3: the norm is exactly 12.  With max_norm 6 the
    applied gradient has norm 6 * 12 / (12 + 1e-6) <= 6; with max_norm 20 the
    gradient is applied unchanged."""
    n = 16
    for max_norm, expect_norm in [(6.0, 6.0 * 12 / (12 + 1e-6)), (20.0, 12.0)]:
        hp = O.hparams(lr=0.0, betas=(0.9, 0.999), max_grad_norm=max_norm)
        st = O.scaler(1.0)
        master, m, v, p16 = _state(n)
        _, d = orc.step(hp, st, [_h(np.full(n, 3.0))], F16, master, m, v, p16, F16, 1.0)
        assert d.norm == 12.0
        applied = m.astype(np.float64) / 0.1          # m = (1 - b1) g_applied
        got = np.linalg.norm(applied)
        assert abs(got - expect_norm) <= 1e-6 * expect_norm, (got, expect_norm)
        assert got <= max_norm * (1 + 1e-6)


# ---------------------------------------------------------------- overflow / scale

_INF16, _NINF16, _NAN16 = 0x7C00, 0xFC00, 0x7E00


def pin_overflow_skips(orc):
    """+inf, -inf, NaN, and +inf with -inf in one element (sum NaN) all skip
    the step: nothing moves, the scale halves, the counter does not advance."""
    n = 16
    base = [_h(np.linspace(-3, 3, n) * 64) for _ in range(2)]
    hp = O.hparams(lr=1e-3, dynamic_scale=True)
    for inject in [[(0, _INF16)], [(1, _NINF16)], [(0, _NAN16)],
                   [(0, _INF16), (1, _NINF16)]]:
        bufs = [b.copy() for b in base]
        for r, val in inject:
            bufs[r][5] = val
        st = O.scaler(64.0)
        st.clean, st.t = 7, 3
        p0 = np.linspace(-1, 1, n).astype(np.float32)
        master, m, v, p16 = _state(n, p0)
        m[:] = 0.5
        v[:] = 0.25
        p16[:] = 123
        own, d = orc.step(hp, st, bufs, F16, master, m, v, p16, F16, 2.0)
        assert own.nonfinite == 1 and d.skip == 1
        assert (master.view(np.uint32) == p0.view(np.uint32)).all()
        assert (m == 0.5).all() and (v == 0.25).all() and (p16 == 123).all()
        assert st.as_tuple() == (32.0, 0, 3, 1, 1)


def pin_no_false_overflow(orc):
    """Largest finite fp16 gradients in two buffers sum to a finite binary32."""
    bufs = [_h(np.full(4, 65504.0)), _h(np.full(4, 65504.0))]
    s = orc.reduce(bufs, F16)
    assert (s == 131008.0).all()
    assert orc.stats_of(s).nonfinite == 0


def pin_loss_scale_tiny_schedule(orc):
    rows = read_golden("loss_scale_tiny.txt")
    hp = O.hparams(dynamic_scale=True, scale_window=1000, min_scale=1.0)
    st = O.scaler(2048.0)
    for step, used, skipped, t_after, after in rows:
        stats = O.Stats(1.0, 1 if int(skipped) else 0, 0)
        d = orc.decide(hp, st, stats, 4.0)
        assert d.scale_used == float(used) and d.skip == int(skipped)
        assert st.t == int(t_after) and st.scale == float(after), step


def pin_loss_scale_window(orc):
    rows = read_golden("loss_scale_window3.txt")
    hp = O.hparams(dynamic_scale=True, scale_window=3, min_scale=1.0)
    st = O.scaler(2.0)
    for step, ev, used, after, clean in rows:
        stats = O.Stats(1.0, 1 if ev == "O" else 0, 0)
        d = orc.decide(hp, st, stats, 1.0)
        assert d.scale_used == float(used), step
        assert st.scale == float(after) and st.clean == int(clean), step


def pin_loss_scale_periodic_overflow(orc):
    """Initial scale 2^16 (initial_scale_power 16), window 1000, an overflow every
    50 steps: the scale is 2^(16-k) after k overflows and never rises."""
    hp = O.hparams(dynamic_scale=True, scale_window=1000)
    st = O.scaler(2.0 ** 16)
    k = 0
    for step in range(1, 201):
        over = step % 50 == 0
        d = orc.decide(hp, st, O.Stats(1.0, int(over), 0), 1.0)
        assert d.scale_used == 2.0 ** (16 - k)
        k += over
    assert st.scale == 2.0 ** 12 and st.t == 196 and st.skipped_total == 4


def pin_static_scale(orc):
    """A fixed scale still skips an overflowing step but never changes."""
    hp = O.hparams(dynamic_scale=False, scale_window=2)
    st = O.scaler(1024.0)
    for over in [0, 0, 1, 0, 0, 0]:
        orc.decide(hp, st, O.Stats(1.0, over, 0), 1.0)
    assert st.scale == 1024.0 and st.t == 5 and st.skipped_total == 1


# ---------------------------------------------------------------- reduction, shards

def pin_accumulation_single_nonzero(orc):
    """R*K buffers that are zero except one give exactly the one-buffer step."""
    n = 32
    x = synth.normal_np(7, 1, 0, n, 0.5, synth.F16)
    hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=0.1)
    p0 = synth.normal_np(7, 2, 0, n, 0.02, synth.F32)
    outs = []
    for bufs in ([x], [np.zeros(n, np.uint16)] * 4 + [x] + [np.zeros(n, np.uint16)]):
        st = O.scaler(8.0)
        master, m, v, p16 = _state(n, p0)
        for _ in range(3):
            orc.step(hp, st, bufs, F16, master, m, v, p16, F16, 6.0)
        outs.append((master.copy(), m.copy(), v.copy(), p16.copy()))
    for a, b in zip(*outs):
        assert (a.view(np.uint8) == b.view(np.uint8)).all()


def pin_accumulation_k_way_sum(orc):
    """K = 4 micro-step buffers holding x/4 sum exactly to x ([CSDN] §2.3:
    the accumulated gradient equals the big-batch gradient)."""
    n = 32
    x = _h(np.arange(-16, 16) * 0.25)
    quarter = _h(_f(x) / 4)
    assert (4 * _f(quarter) == _f(x)).all()
    s1 = orc.reduce([x], F16)
    s4 = orc.reduce([quarter] * 4, F16)
    assert (s1 == s4).all() and s1.size == n


def pin_reduce_order(orc):
    """Buffers are summed in index order in binary32: 2^24 + 1 + 1 rounds twice
    to 2^24 in that order (fp32 ties-to-even), but 1 + 1 + 2^24 = 2^24 + 2."""
    big = np.array([0x4B80], np.uint16)        # bf16 2^24
    one = np.array([0x3F80], np.uint16)        # bf16 1.0
    assert orc.f16_to_f32(big, BF16)[0] == 2.0 ** 24
    assert orc.reduce([big, one, one], BF16)[0] == 2.0 ** 24
    assert orc.reduce([one, one, big], BF16)[0] == 2.0 ** 24 + 2


def pin_union_of_shards(orc):
    """N shard steps with the rank-order fold of their statistics equal one
    unsharded step over the same buffers ([CSDN] §2.4: each GPU updates its
    own slice; [ALGO]: reduce-scatter, local update, all-gather)."""
    numel, N, R = 1003, 4, 4
    for max_norm in (0.0, 1e-3):
        _, _, S, P = orc.shard_bounds(numel, N, 0)
        grads = [np.zeros(P, np.uint16) for _ in range(R)]
        for r in range(R):
            grads[r][:numel] = synth.normal_np(1, 1 + r, 0, numel, 1e-3 * 2048, synth.F16)
        p0 = synth.normal_np(1, 0, 0, numel, 0.02, synth.F32)
        hp = O.hparams(lr=1e-3, max_grad_norm=max_norm, dynamic_scale=True)
        # unsharded
        st = O.scaler(2048.0)
        ref = _state(numel, p0)
        for _ in range(3):
            orc.step(hp, st, [g[:numel].copy() for g in grads], F16, *ref, F16, float(R))
        # sharded
        states = [O.scaler(2048.0) for _ in range(N)]
        shards = []
        for r in range(N):
            b, e, _, _ = orc.shard_bounds(numel, N, r)
            shards.append((b, e, _state(e - b, p0[b:e])))
        for _ in range(3):
            per = [orc.stats_of(orc.reduce([g[b:e].copy() for g in grads], F16))
                   for b, e, _ in shards]
            G = orc.fold_stats(per)
            for r, (b, e, bufs) in enumerate(shards):
                orc.step(hp, states[r], [g[b:e].copy() for g in grads], F16, *bufs, F16,
                         float(R), G)
        for i in range(4):
            cat = np.concatenate([sh[2][i] for sh in shards])
            if max_norm == 0.0:
                assert (cat.view(np.uint8) == ref[i].view(np.uint8)).all(), i
            else:
                if i == 3:
                    d = np.abs(cat.astype(np.int32) - ref[i].astype(np.int32))
                    assert d.max() <= 1
                else:
                    _close(cat, ref[i], 1e-6, 1e-9)
        assert all(s.as_tuple() == st.as_tuple() for s in states)




def pin_global_overflow_across_shards(orc):
    """An overflow in any one shard skips the step on every rank: the scalar
    all-reduce ORs the flags and sums the squares in rank order."""
    per = [O.Stats(1.0, 0, 0), O.Stats(2.0, 1, 0), O.Stats(0.5, 0, 0)]
    G = orc.fold_stats(per)
    assert G.nonfinite == 1 and G.sumsq == 3.5
    assert orc.fold_stats([O.Stats(1.0, 0, 0), O.Stats(0.25, 0, 0)]).nonfinite == 0
    numel, N = 40, 4
    grads = [synth.normal_np(9, 1, 0, numel, 4.0, synth.F16)]
    grads[0][27] = _INF16                      # lands in shard 2
    hp = O.hparams(lr=1e-3, dynamic_scale=True)
    per, shards = [], []
    for r in range(N):
        b, e, _, _ = orc.shard_bounds(numel, N, r)
        per.append(orc.stats_of(orc.reduce([grads[0][b:e].copy()], F16)))
        shards.append((b, e))
    G = orc.fold_stats(per)
    for r, (b, e) in enumerate(shards):
        st = O.scaler(16.0)
        master, m, v, p16 = _state(e - b, np.ones(e - b))
        _, d = orc.step(hp, st, [grads[0][b:e].copy()], F16, master, m, v, p16, F16, 1.0, G)
        assert d.skip == 1 and (master == 1.0).all() and st.scale == 8.0, r




def pin_sum_of_squares_is_correctly_rounded(orc):
    """The sum of squares equals math.fsum (the correctly rounded sum) of the
    exact binary64 squares, to within one ulp, for sums with a wide dynamic
    range and many terms."""
    import math
    rng = np.random.default_rng(8)
    for n, spread in [(10_000, 2), (200_000, 30), (3, 60)]:
        s = (rng.standard_normal(n) * 2.0 ** rng.integers(-spread, spread, n)).astype(np.float32)
        got = orc.stats_of(s).sumsq
        ref = math.fsum((s.astype(np.float64) ** 2).tolist())
        assert abs(got - ref) <= math.ulp(ref), (n, got, ref)
    # a case where plain sequential binary64 summation loses the small terms
    s = np.array([2.0 ** 30] + [2.0 ** -1] * 4096, np.float32)
    assert orc.stats_of(s).sumsq == 2.0 ** 60 + 4096 * 0.25




def pin_consolidation_is_the_unsharded_state(orc):
    """zero_to_fp32 of a sharded run equals the master weights of the same run
    done unsharded; padding never appears in the result."""
    numel, N = 1001, 4
    grads = [synth.normal_np(21, 1 + r, 0, numel, 8.0, synth.F16) for r in range(2)]
    p0 = synth.normal_np(21, 0, 0, numel, 0.02, synth.F32)
    hp = O.hparams(lr=1e-3)
    ref = _state(numel, p0)
    orc.step(hp, O.scaler(4.0), grads, F16, *ref, F16, 2.0)
    bounds = [orc.shard_bounds(numel, N, r) for r in range(N)]
    G = orc.fold_stats([orc.stats_of(orc.reduce([g[b:e].copy() for g in grads], F16))
                        for b, e, _, _ in bounds])
    shards = []
    for b, e, _, _ in bounds:
        st = _state(e - b, p0[b:e])
        orc.step(hp, O.scaler(4.0), [g[b:e].copy() for g in grads], F16, *st, F16, 2.0, G)
        shards.append(st[0])
    full = orc.consolidate(shards, numel)
    assert full.size == numel
    assert (full.view(np.uint32) == ref[0].view(np.uint32)).all()




def pin_hysteresis_schedule(orc):
    """Hysteresis 2 (tests/golden/loss_scale_hysteresis2.txt); hysteresis 1 is
    the halve-on-every-overflow rule of the other schedules."""
    rows = read_golden("loss_scale_hysteresis2.txt")
    hp = O.hparams(dynamic_scale=True, scale_window=3, min_scale=1.0, hysteresis=2)
    st = O.scaler(8.0)
    for step, ev, used, after, ovf in rows:
        d = orc.decide(hp, st, O.Stats(1.0, 1 if ev == "O" else 0, 0), 1.0)
        assert d.scale_used == float(used), step
        assert st.scale == float(after) and st.overflows == int(ovf), step
    hp1 = O.hparams(dynamic_scale=True, scale_window=1000, hysteresis=1)
    st = O.scaler(64.0)
    for k in range(4):
        orc.decide(hp1, st, O.Stats(1.0, 1, 0), 1.0)
        assert st.scale == 64.0 / 2 ** (k + 1)


def pin_warmup_lr(orc):
    """WarmupLR with the ds_config.json values ("DeepSpeed tutorial" §3.2:
    warmup_min_lr 0, warmup_max_lr 2e-5, warmup_num_steps 1000), read as a
    linear rise over the updates: update t uses 2e-5 * min(t, 1000) / 1000.
    Skipped steps do not advance it (§2.4: the scheduler steps with every
    parameter update); with 0 steps the configured lr is used."""
    hp = O.hparams(lr=5.0, weight_decay=0.5, warmup=(0.0, 2e-5, 1000))
    st = O.scaler(1.0)
    seen = {}
    for k in range(1, 1203):
        over = (k % 300 == 0)
        d = orc.decide(hp, st, O.Stats(1.0, int(over), 0), 1.0)
        if not over:
            seen[st.t] = (d.lr, d.decay)
    assert seen[1][0] == 2e-5 * 1 / 1000
    assert seen[500][0] == 2e-5 * 500 / 1000
    assert seen[1000][0] == 2e-5 and seen[1198][0] == 2e-5
    assert seen[1][1] == np.float32(1.0 - 2e-8 * 0.5)
    hp0 = O.hparams(lr=3e-4, warmup=(0.0, 2e-5, 0))
    assert orc.decide(hp0, O.scaler(1.0), O.Stats(1.0, 0, 0), 1.0).lr == 3e-4
    # first update of a warm-up run: the bias-corrected step moves by
    # -lr_1 * g / (|g| + eps) with lr_1 = max / T
    hpw = O.hparams(warmup=(1e-3, 1e-2, 4))
    master, m, v, p16 = _state(8)
    bufs = [_h(_G8)]
    g = _f(bufs[0])
    orc.step(hpw, O.scaler(1.0), bufs, F16, master, m, v, p16, F16, 1.0)
    _close(master, -(1e-3 + 9e-3 / 4) * g / (np.abs(g) + 1e-8), 2e-6)


def _m16_step(orc, p16_bits, lr, dtype, steps=1, fp32_master=False):
    """`steps` steps at p with g = 1, beta1 = beta2 = 0, no bias correction,
    wd = 0, scale 1, no clipping: each step is p - lr exactly (m = v = 1 and
    den = 1 + 1e-8 rounds to 1 in binary32), then the 16-bit rounding."""
    hp = O.hparams(lr=lr, betas=(0.0, 0.0), bias_correction=False)
    st = O.scaler(1.0)
    n = p16_bits.size
    p16 = p16_bits.copy()
    master = _f(p16, dtype).astype(np.float32) if fp32_master else None
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    one = np.full(n, 0x3C00 if dtype == F16 else 0x3F80, np.uint16)
    for _ in range(steps):
        orc.step(hp, st, [one], dtype, master, m, v, p16, dtype, 1.0)
    return p16


def pin_low_precision_master(orc):
    """Low-precision master weights (reading R17: no fp32 master array, the
    16-bit parameter is the master).  Closed forms from the formats' rounding
    at p = 1 (each step computes p - lr exactly, see _m16_step):
    bf16: lr 2^-4 gives 0.9375 = 0x3F70 exactly; lr 3*2^-10 gives
    0.9970703125, nearest bf16 1 - 2^-8 = 0x3F7F; lr 2^-10 is within half an
    ulp (2^-9) of 1 and is lost, every step, so 16 steps leave 0x3F80 where an
    fp32 master reaches 1 - 2^-6 = 0x3F7C.  fp16: lr 2^-12 lands exactly
    halfway between 1 and 1 - 2^-11 and ties to even, 0x3C00; lr 2^-10 gives
    1 - 2^-10 = 0x3BFE exactly."""
    one_b = np.array([0x3F80], np.uint16)
    one_h = np.array([0x3C00], np.uint16)
    assert _m16_step(orc, one_b, 2.0 ** -4, BF16)[0] == 0x3F70
    assert _m16_step(orc, one_b, 3 * 2.0 ** -10, BF16)[0] == 0x3F7F
    assert _m16_step(orc, one_b, 2.0 ** -10, BF16, steps=16)[0] == 0x3F80
    assert _m16_step(orc, one_b, 2.0 ** -10, BF16, steps=16, fp32_master=True)[0] == 0x3F7C
    assert _m16_step(orc, one_h, 2.0 ** -12, F16)[0] == 0x3C00
    assert _m16_step(orc, one_h, 2.0 ** -10, F16)[0] == 0x3BFE


def pin_low_precision_master_round_trip(orc):
    """With lr = 0 a low-precision master keeps every finite 16-bit pattern
    (widening is exact and p * 1 - 0 = p), in both formats."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dtype, expmask in ((F16, 0x7C00), (BF16, 0x7F80)):
        fin = codes[(codes & expmask) != expmask]
        hp = O.hparams(lr=0.0, weight_decay=0.0)
        n = fin.size
        p16 = fin.copy()
        g = np.full(n, 0x3C00 if dtype == F16 else 0x3F80, np.uint16)
        orc.step(hp, O.scaler(1.0), [g], dtype, None, np.zeros(n, np.float32),
                 np.zeros(n, np.float32), p16, dtype, 1.0)
        assert (p16 == fin).all()


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
