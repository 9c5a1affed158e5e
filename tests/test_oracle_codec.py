"""Pins for the oracle's E4M3 codec.

The FP8 format is E4M3 (named by the commentary page's "FP8" background box:
4 exponent bits, 3 mantissa bits).  The oracle's encoder/decoder are written
from the OCP 8-bit floating point definition; here they are checked against an
independent implementation, torch's float8_e4m3fn, and against values fixed by
the definition itself (tests/golden/e4m3_points.txt).
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_points.txt")


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_on_all_codes():
    ref = torch_decode_all()
    ours = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2  # 0x7F and 0xFF: E4M3 has no infinities
    assert np.array_equal(ref[~nan], ours[~nan])
    # signed zero is kept
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_golden_points_from_definition():
    """Values the format definition fixes (largest normal, smallest normal and
    subnormal, a few ties)."""
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            v, code = line.split()
            assert oracle.e4m3_encode(float(v)) == int(code, 16), line


def _grid():
    vals = torch_decode_all()
    pos = np.unique(vals[(~np.isnan(vals)) & (vals >= 0)])
    return pos


def test_encode_matches_torch_round_to_nearest_even():
    """Every representable value, every midpoint between neighbours (ties go to
    the even code), one fp32 ulp either side of each midpoint, and random
    magnitudes over the whole range, both signs; inputs pre-clamped to +-448
    because torch's cast is not saturating."""
    pos = _grid()
    mids = (pos[:-1] + pos[1:]) / 2
    pts = [pos, mids]
    m32 = mids.astype(np.float32)
    pts.append(np.nextafter(m32, np.float32(np.inf)).astype(np.float64))
    pts.append(np.nextafter(m32, np.float32(-np.inf)).astype(np.float64))
    rng = np.random.default_rng(0)
    pts.append(np.exp(rng.uniform(np.log(1e-5), np.log(448.0), 200_000)))
    pts.append(rng.uniform(0, 2e-3, 20_000))  # subnormal region
    v = np.concatenate(pts).astype(np.float32)
    v = np.concatenate([v, -v])
    ours = oracle.e4m3_encode_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:10]]


def test_encode_saturates_instead_of_overflowing():
    for v in (448.0, 449.0, 464.0, 480.0, 1e4, 3.0e38, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE


def test_roundtrip_of_every_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c


@pytest.mark.parametrize("s", [1.0, 0.25, 3.0 / 448.0, 1e-3])
def test_quantize_divides_in_fp32(s):
    """q(v; s) = E4M3(fp32(v) / s) with the division in fp32 (not v * (1/s))."""
    rng = np.random.default_rng(1)
    v = rng.standard_normal(5000).astype(np.float32) * 100 * s
    ref = torch.from_numpy((v / np.float32(s)).astype(np.float32)).clamp(-448, 448)
    ref = ref.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.quantize(float(a), s) for a in v], np.uint8)
    assert np.array_equal(ours, ref)
