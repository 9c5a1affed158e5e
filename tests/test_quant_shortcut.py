"""The kernels take the E4M3 code of fl32(v / s) from q = fl32(v * fl32(1 / s))
unless q lies within 8 ulp of an E4M3 rounding midpoint (the 20 mantissa bits
below E4M3's three are near 0x80000) or in E4M3's subnormal range, where they
divide.  This checks the argument on the host: wherever the shortcut is
taken, q and the rounded quotient have the same code (the oracle's encoder),
on random values and on values placed next to every midpoint."""
import numpy as np

import oracle


def _shortcut_taken(q):
    b = q.view(np.uint32) & np.uint32(0x7FFFFFFF)
    d = (b & np.uint32(0xFFFFF)).astype(np.int64) - 0x80000
    return (b == 0) | (((b >> 23) >= 121) & (np.abs(d) > 8))


def _check(v, s):
    v = v.astype(np.float32)
    s = np.float32(s)
    rs = np.float32(1.0) / s
    q = (v * rs).astype(np.float32)
    exact = (v / s).astype(np.float32)
    fast = _shortcut_taken(q)
    assert fast.mean() > 0.5
    codes_q = oracle.e4m3_encode_array(q[fast])
    codes_e = oracle.e4m3_encode_array(exact[fast])
    assert np.array_equal(codes_q, codes_e)


def test_shortcut_random_values():
    rng = np.random.default_rng(7)
    for _ in range(8):
        amax = np.float32(np.exp(rng.uniform(-15, 15)))
        s = np.float32(amax / np.float32(448.0))
        v = np.clip(rng.standard_normal(200_000) * amax / 3, -amax, amax)
        _check(v, s)


def test_shortcut_next_to_every_midpoint():
    rng = np.random.default_rng(8)
    mids = np.array([(m + 0.5) * 2.0 ** (e - 3) for e in range(-6, 9) for m in range(8, 16)])
    for _ in range(8):
        s = np.float32(np.exp(rng.uniform(-10, 10)))
        t = rng.choice(mids, 200_000) * (1 + rng.integers(-40, 41, 200_000) * 2.0 ** -24)
        v = (t * s).astype(np.float32)
        v = v[np.abs(v / s) <= 448]
        _check(v, s)
