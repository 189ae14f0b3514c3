"""Sharded checkpoint files on the host: round trip, corruption detection and
zero_to_fp32 consolidation against the oracle's definition."""
import os

import numpy as np
import pytest

import oracle as O
import synth


@pytest.fixture(scope="module")
def z():
    from zero_sharded_mixed_05_gb300 import _build
    _build.build()
    import zero_sharded_mixed_05_gb300 as z
    return z


def _info(z, numel, world, rank, scale=1024.0, t=7):
    b, e, _, _ = O.shard_bounds(numel, world, rank)
    sc = z.zero_opt_scaler_state(scale, 1, 3, t, 2)
    return z.zero_opt_ckpt_info(numel, world, rank, b, e - b, sc)


def test_round_trip_is_bit_exact(z, tmp_path):
    numel, world = 1_000_003, 4
    for rank in range(world):
        info = _info(z, numel, world, rank)
        n = info.real_len
        arrs = [synth.normal_np(3, k, rank * n, n, 0.5, synth.F32) for k in range(3)]
        path = str(tmp_path / f"s{rank}.bin")
        z.zero_opt_ckpt_write(path, info, *arrs)
        got, *back = z.zero_opt_ckpt_read(path)
        assert (got.numel, got.world, got.rank, got.begin, got.real_len) == \
            (numel, world, rank, info.begin, n)
        assert got.scaler.as_tuple() == info.scaler.as_tuple()
        for a, b in zip(arrs, back):
            assert (a.view(np.uint32) == b.view(np.uint32)).all()
        assert os.path.getsize(path) == 96 + 12 * n   # header: 8+4+4+8+4+4+8+8+4+4+8+8+8+4+4+8


def test_corruption_is_detected(z, tmp_path):
    info = _info(z, 1001, 2, 1)
    arrs = [np.arange(info.real_len, dtype=np.float32) * k for k in range(3)]
    path = str(tmp_path / "s.bin")
    z.zero_opt_ckpt_write(path, info, *arrs)
    raw = bytearray(open(path, "rb").read())
    flipped = bytearray(raw)
    flipped[200] ^= 0x10
    open(path, "wb").write(flipped)
    with pytest.raises(z.ZeroOptError, match="checksum"):
        z.zero_opt_ckpt_read(path)
    open(path, "wb").write(raw[:-4])
    with pytest.raises(z.ZeroOptError, match="size"):
        z.zero_opt_ckpt_read(path)
    bad = bytearray(raw)
    bad[0:8] = b"NOTASHRD"
    open(path, "wb").write(bad)
    with pytest.raises(z.ZeroOptError, match="not a shard"):
        z.zero_opt_ckpt_read(path)


def test_inconsistent_info_is_rejected(z, tmp_path):
    info = _info(z, 1001, 4, 2)
    a = np.zeros(info.real_len, np.float32)
    info.begin += 1
    with pytest.raises(z.ZeroOptError):
        z.zero_opt_ckpt_write(str(tmp_path / "x.bin"), info, a, a, a)
    info = _info(z, 1001, 4, 2)
    info.rank = 4
    with pytest.raises(z.ZeroOptError):
        z.zero_opt_ckpt_write(str(tmp_path / "x.bin"), info, a, a, a)


def test_consolidation_matches_the_oracle(z, tmp_path):
    """Shard files of an oracle-stepped sharded run (written in shuffled order)
    consolidate to the oracle's zero_to_fp32 and to its unsharded run."""
    numel, world = 50_003, 4
    grads = [synth.normal_np(5, 1 + r, 0, numel, 4.0, synth.F16) for r in range(2)]
    p0 = synth.normal_np(5, 0, 0, numel, 0.02, synth.F32)
    hp = O.hparams(lr=1e-3, weight_decay=0.01)
    bounds = [O.shard_bounds(numel, world, r) for r in range(world)]
    G = O.fold_stats([O.stats_of(O.reduce([g[b:e].copy() for g in grads], O.FP16))
                      for b, e, _, _ in bounds])
    shards, paths = [], []
    for r in (2, 0, 3, 1):
        b, e, _, _ = bounds[r]
        st = (p0[b:e].copy(), np.zeros(e - b, np.float32), np.zeros(e - b, np.float32),
              np.zeros(e - b, np.uint16))
        sc = O.scaler(4.0)
        O.step(hp, sc, [g[b:e].copy() for g in grads], O.FP16, *st, O.FP16, 2.0, G)
        info = _info(z, numel, world, r, scale=sc.scale, t=sc.t)
        path = str(tmp_path / f"rank{r}.bin")
        z.zero_opt_ckpt_write(path, info, st[0], st[1], st[2])
        paths.append(path)
        shards.append((r, st[0]))
    full = z.zero_opt_consolidate_fp32(paths, numel)
    ref = O.consolidate([a for _, a in sorted(shards)], numel)
    assert (full.view(np.uint32) == ref.view(np.uint32)).all()
    un = (p0.copy(), np.zeros(numel, np.float32), np.zeros(numel, np.float32),
          np.zeros(numel, np.uint16))
    O.step(hp, O.scaler(4.0), grads, O.FP16, *un, O.FP16, 2.0)
    assert (full.view(np.uint32) == un[0].view(np.uint32)).all()
    # a missing or duplicated rank is an error
    with pytest.raises(z.ZeroOptError):
        z.zero_opt_consolidate_fp32(paths[:3], numel)
    with pytest.raises(z.ZeroOptError):
        z.zero_opt_consolidate_fp32([paths[0]] * 4, numel)
    with pytest.raises(z.ZeroOptError):
        z.zero_opt_consolidate_fp32(paths, numel + 1)
