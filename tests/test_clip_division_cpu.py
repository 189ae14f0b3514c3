"""The decision divides max_norm by b = norm + 1e-6 only when max_norm < b.

The clip coefficient is min(1, max_norm / b) in binary64 (rounded to
nearest).  The decision code skips the division when max_norm >= b and takes
1; that is the same value only because, for binary64 m and b, m >= b gives a
rounded quotient of at least 1 and m < b one below 1.  These tests hold the
second half at its tightest cases (m one unit below b in b's last place, b a
power of two, subnormal and huge operands) and the first half at m == b and
just above, with IEEE division as numpy performs it.
"""
import numpy as np


def _clip_plain(m, b):
    q = np.float64(m) / np.float64(b)
    return np.float64(1.0) if q > 1.0 else q


def _clip_shortcut(m, b):
    return np.float64(1.0) if not (m < b) else np.float64(m) / np.float64(b)


def _check(m, b):
    m, b = np.float64(m), np.float64(b)
    p, s = _clip_plain(m, b), _clip_shortcut(m, b)
    assert p.tobytes() == s.tobytes(), (m, b, p, s)
    if m < b:
        assert np.float64(m) / np.float64(b) < 1.0, (m, b)


def test_one_unit_below_b_rounds_below_one():
    rng = np.random.default_rng(0x5EED0C11)
    exps = rng.integers(-1000, 1000, size=20000)
    mant = rng.uniform(1.0, 2.0, size=20000)
    for e, f in zip(exps, mant):
        b = np.ldexp(np.float64(f), int(e))
        m = np.nextafter(b, np.float64(0.0))
        _check(m, b)
        _check(np.nextafter(m, np.float64(0.0)), b)


def test_powers_of_two_and_extremes():
    for e in range(-1074, 1024):
        b = np.ldexp(np.float64(1.0), e)
        _check(np.nextafter(b, np.float64(0.0)), b)
        _check(b, b)
        _check(np.nextafter(b, np.float64(np.inf)), b)
    big = np.finfo(np.float64).max
    _check(np.nextafter(big, 0.0), big)
    _check(np.float64(5e-324), np.float64(1e-323))


def test_equal_and_above_give_one():
    rng = np.random.default_rng(0x5EED0C12)
    for b in rng.uniform(1e-7, 1e4, size=20000):
        _check(b, b)
        _check(np.nextafter(b, np.inf), b)
        _check(b * 3.0, b)


def test_the_usual_range_of_norms():
    # max_norm 1.0 against norms around it, as the clipped configurations see
    rng = np.random.default_rng(0x5EED0C13)
    for norm in np.concatenate([rng.uniform(0.0, 2.0, 20000), [0.0, 1.0 - 1e-6, 1.0]]):
        b = np.float64(norm) + np.float64(1e-6)
        _check(np.float64(1.0), b)
