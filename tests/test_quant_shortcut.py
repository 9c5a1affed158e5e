"""The kernels take the E4M3 code of fl32(v / s) from two bracketing products:
with rs = fl32(1 / s), rlo = fl32(rs (1 - 2^-20)) and rhi = fl32(rs (1 + 2^-20)),
fl32(v rlo) and fl32(v rhi) lie on either side of the rounded quotient, so when
both have the same code (the encoder is monotonic) the quotient has it too;
otherwise the kernel divides.  This checks the argument on the host with the
oracle's encoder: wherever the two codes agree they equal the quotient's code,
on random values over 30 decades of scale and on values placed next to every
E4M3 rounding midpoint, subnormal ones included.  A bracket without the margin
(rlo = rhi = rs, the plain reciprocal multiply) fails the midpoint case, and a
scale whose reciprocal overflows brackets nothing."""
import numpy as np

import oracle

MARGIN = 2.0 ** -20


def _codes(v, s, margin):
    """(codes of fl32(v rlo), codes of fl32(v rhi), codes of fl32(v / s))."""
    v = v.astype(np.float32)
    s = np.float32(s)
    rs = np.float32(1.0) / s
    rlo = np.float32(rs * np.float32(1 - margin))
    rhi = np.float32(rs * np.float32(1 + margin))
    enc = oracle.e4m3_encode_array
    return enc((v * rlo).astype(np.float32)), enc((v * rhi).astype(np.float32)), \
        enc((v / s).astype(np.float32))


def _agree_where_fast(v, s, margin=MARGIN):
    lo, hi, exact = _codes(v, s, margin)
    fast = lo == hi
    return fast.mean(), bool(np.array_equal(lo[fast], exact[fast]))


def _next_to_midpoints(rng, s, n):
    normal = [(m + 0.5) * 2.0 ** (e - 3) for e in range(-6, 9) for m in range(8, 16)]
    subnormal = [(k + 0.5) * 2.0 ** -9 for k in range(8)]
    mids = np.array(normal + subnormal)
    t = rng.choice(mids, n) * (1 + rng.integers(-40, 41, n) * 2.0 ** -24)
    v = (t * s).astype(np.float32)
    return v[np.abs(v / s) <= 448]


def test_bracket_random_values():
    rng = np.random.default_rng(7)
    for _ in range(8):
        amax = np.float32(np.exp(rng.uniform(-15, 15)))
        s = np.float32(amax / np.float32(448.0))
        v = np.clip(rng.standard_normal(200_000) * amax / 3, -amax, amax)
        frac, ok = _agree_where_fast(v, s)
        assert ok
        assert frac > 0.999


def test_bracket_next_to_every_midpoint():
    rng = np.random.default_rng(8)
    for _ in range(8):
        s = np.float32(np.exp(rng.uniform(-10, 10)))
        frac, ok = _agree_where_fast(_next_to_midpoints(rng, s, 200_000), s)
        assert ok
        assert frac > 0.5


def test_bracket_without_margin_fails_at_midpoints():
    rng = np.random.default_rng(8)
    bad = 0
    for _ in range(8):
        s = np.float32(np.exp(rng.uniform(-10, 10)))
        _, ok = _agree_where_fast(_next_to_midpoints(rng, s, 200_000), s, margin=0.0)
        bad += not ok
    assert bad > 0


def test_overflowing_reciprocal_brackets_nothing():
    # s below 2^-128: 1/s overflows; the kernels then bracket with (0, inf),
    # whose codes differ for every v (zero: 0 against NaN), so they divide
    s = np.float32(2.0 ** -130)
    v = np.array([0.0, 1e-40, -3e-39, 2.0 ** -135], np.float32)
    enc = oracle.e4m3_encode_array
    with np.errstate(invalid="ignore", over="ignore"):
        assert np.isinf(np.float32(1.0) / s)
        lo = enc((v * np.float32(0.0)).astype(np.float32))
        hi = enc((v * np.float32(np.inf)).astype(np.float32))
    assert np.all(lo != hi)
