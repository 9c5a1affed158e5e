"""Pins for the oracle's dynamic per-tensor activation quantisation.

FP8 per-tensor scaling is the step of section "Backend routing for FP8 tensor
quantization" (English original page); the format is E4M3 (the commentary
page's "FP8" box).  The oracle reads it as s = amax|x| / 448 in fp32 (1 when
x is all zero) and code = E4M3_rne_satfinite(fp32(x) / s) with an IEEE fp32
division.  Here the same quantities are rebuilt from independent pieces:
numpy's float32 reduction and elementwise division, and torch's own
float8_e4m3fn cast (inputs clamped to +-448 first, because torch's cast does
not saturate).  A slip in the oracle (amax over the wrong length or taken
after a conversion, a reciprocal instead of the division, a wrong zero rule)
fails one of these cases.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_align_gb300 import inputs


def independent_quantize(xb: torch.Tensor):
    """(codes uint8, s fp32) of a bf16 tensor without the oracle's code."""
    xf = xb.float().numpy().astype(np.float32)
    amax = np.float32(np.abs(xf).max()) if xf.size else np.float32(0)
    s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
    q = (xf / np.full_like(xf, s)).astype(np.float32)  # IEEE fp32, elementwise
    q = np.clip(q, -448.0, 448.0)
    codes = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, float(s)


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("shape,amp,seed", [
    ((1, 16), 1.0, 0), ((7, 2048), 1.0, 1), ((3, 4097), 30.0, 2), ((64, 4096), 1e-3, 3),
    ((5, 333), 1e4, 4), ((1,), 2.5, 5), ((2, 3, 40), 0.2, 6),
])
def test_random_tensors_match_independent_quantisation(shape, amp, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(*shape, generator=g) * amp).to(torch.bfloat16)
    codes, s = oracle.quantize_act(x)
    ref_codes, ref_s = independent_quantize(x)
    assert s == ref_s
    assert codes.shape == x.shape
    assert np.array_equal(codes, ref_codes)


def test_all_zero_tensor_has_scale_one_and_zero_codes():
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    codes, s = oracle.quantize_act(x)
    assert s == 1.0
    assert np.all(codes == 0)
    # negative zeros keep their sign bit
    codes, s = oracle.quantize_act(-x)
    assert s == 1.0 and np.all(codes == 0x80)


def test_single_nonzero_maps_to_the_largest_code():
    """amax is that one element: it becomes exactly +-448 (code 0x7E / 0xFE)."""
    for v in (3.0, -0.0078125, 1.5e3):
        a = np.zeros(100, np.float32)
        a[37] = v
        x = _bf16(a)
        codes, s = oracle.quantize_act(x)
        assert s == np.float32(abs(np.float32(x[37].item())) / np.float32(448.0))
        assert codes[37] == (0xFE if v < 0 else 0x7E)
        assert np.all(np.delete(codes, 37) == 0)


def test_amax_spans_the_whole_tensor():
    """The largest magnitude sits in the last element: a scale taken over a
    shorter length would differ."""
    a = np.full(1000, 0.5, np.float32)
    a[-1] = -64.0
    codes, s = oracle.quantize_act(_bf16(a))
    assert s == np.float32(64.0) / np.float32(448.0)
    assert codes[-1] == 0xFE
    ref_codes, _ = independent_quantize(_bf16(a))
    assert np.array_equal(codes, ref_codes)


def test_scale_equals_the_layer_oracles_s_x():
    """The whole-layer oracle quantises x with the same rule."""
    w = inputs.make_weights(128, 128, 4, "fp8", seed=3)
    a = inputs.make_activations(11, 128, 4, "uniform", seed=3)
    ref = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, 2, True)
    _, s = oracle.quantize_act(a.x)
    assert s == ref["s_x"]
    assert s == independent_quantize(a.x)[1]


@pytest.mark.parametrize("amax_bits", [0x3FA3, 0x3FC6, 0x4000, 0x42E0, 0x3C00])
def test_every_bf16_value_up_to_amax(amax_bits):
    """Every finite bf16 magnitude up to amax, both signs, with amax itself in
    the tensor.  With these amax values some quotients land where a multiply
    by the rounded reciprocal 1/s would pick another code than the division
    (found by exhaustive search), so the division rule is pinned too."""
    mags = (np.arange(0, amax_bits + 1, dtype=np.uint32) << 16).view(np.float32)
    a = np.concatenate([mags, -mags])
    x = _bf16(a)
    codes, s = oracle.quantize_act(x)
    ref_codes, ref_s = independent_quantize(x)
    assert s == ref_s
    assert np.array_equal(codes, ref_codes)
