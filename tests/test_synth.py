"""The seeded input generator: definition, slicing and distribution."""
import numpy as np

import synth


def _scalar_reference(seed, stream, j, sigma):
    k = synth.key(seed, stream)
    acc = 0
    for u in range(12):
        d = synth.mix64_int(k + (12 * j + u + 1) * synth.GAMMA)
        acc += d >> 40
    return ((acc - 6 * (1 << 24)) * 2.0 ** -24) * sigma


def test_matches_definition():
    vals = synth.normal_f64_np(0x5EED0001, 3, 100, 5, 2.5)
    for i, v in enumerate(vals):
        assert v == _scalar_reference(0x5EED0001, 3, 100 + i, 2.5)


def test_splitmix_known_value():
    # SplitMix64 seeded with 0: the first output of next() is the output
    # function applied to 0x9E3779B97F4A7C15.
    assert synth.mix64_int(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_offsets_are_slices():
    a = synth.normal_np(7, 1, 0, 1000, 1.0, synth.F32)
    b = synth.normal_np(7, 1, 300, 200, 1.0, synth.F32)
    assert (a[300:500] == b).all()


def test_kinds_round_the_same_values():
    x64 = synth.normal_f64_np(9, 2, 0, 4096, 3e-2)
    f32 = synth.normal_np(9, 2, 0, 4096, 3e-2, synth.F32)
    f16 = synth.normal_np(9, 2, 0, 4096, 3e-2, synth.F16)
    assert (f32 == x64.astype(np.float32)).all()
    assert (f16 == f32.astype(np.float16).view(np.uint16)).all()
    bf = synth.normal_np(9, 2, 0, 4096, 3e-2, synth.BF16)
    assert bf.dtype == np.uint16


def test_distribution():
    x = synth.normal_f64_np(1, 0, 0, 1 << 18, 1.0)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.abs(x).max() <= 6.0


def test_streams_differ():
    a = synth.normal_np(1, 0, 0, 64, 1.0, synth.F32)
    b = synth.normal_np(1, 1, 0, 64, 1.0, synth.F32)
    c = synth.normal_np(2, 0, 0, 64, 1.0, synth.F32)
    assert not (a == b).all() and not (a == c).all()


def test_seeded_indices_in_range():
    idx = synth.seeded_indices(5, 77, 100, 10, 20)
    assert all(10 <= i < 20 for i in idx) and len(set(idx)) > 3
