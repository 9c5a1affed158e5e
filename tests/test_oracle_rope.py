"""Pins of the oracle's inverse rotary embedding + per-head FP8 quantisation.

The pages only name the fused kernel (rotary position embedding with FP8
quantisation, per head); the oracle's reading is RoFormer's rotation of the
pairs (2i, 2i+1) by the negated angle, then one E4M3 scale per head over all
tokens.  These checks pin that reading with formulations independent of the
oracle's code: complex multiplication by exp(-i angle), exact special angles,
rotation invariants, and the per-head scale against torch's float8 cast.
"""
import numpy as np
import torch

import oracle
from mixture_experts_layer_align_gb300 import inputs


def _run(T=37, NH=6, D=64, max_pos=512, seed=0):
    r = inputs.make_rope_inputs(T, NH, D, max_pos, seed=seed)
    return r, oracle.inv_rope_quant(r.x, r.positions, r.cos, r.sin)


def test_rotation_is_complex_multiplication_by_the_negated_angle():
    r, o = _run()
    x = r.x.float().numpy().astype(np.float64)
    z = x[..., 0::2] + 1j * x[..., 1::2]
    pos = r.positions.numpy()
    c = r.cos.numpy().astype(np.float64)[pos][:, None, :]
    s = r.sin.numpy().astype(np.float64)[pos][:, None, :]
    w = z * (c - 1j * s)  # e^{-i angle}
    y = o["y"].astype(np.float64)
    np.testing.assert_allclose(y[..., 0::2], w.real, rtol=0, atol=1e-6 * np.abs(x).max())
    np.testing.assert_allclose(y[..., 1::2], w.imag, rtol=0, atol=1e-6 * np.abs(x).max())


def test_special_angles_are_exact():
    T, NH, D = 5, 2, 8
    r = inputs.make_rope_inputs(T, NH, D, 4, seed=3)
    cos = torch.tensor([[1.0] * 4, [0.0] * 4, [-1.0] * 4, [0.0] * 4])
    sin = torch.tensor([[0.0] * 4, [1.0] * 4, [0.0] * 4, [-1.0] * 4])
    pos = torch.tensor([0, 1, 2, 3, 1], dtype=torch.int32)
    y = oracle.inv_rope_quant(r.x, pos, cos, sin)["y"]
    x = r.x.float().numpy()
    x0, x1 = x[..., 0::2], x[..., 1::2]
    for t, p in enumerate(pos.tolist()):
        # angle 0: identity; pi/2 (inverse turns by -pi/2): (x1, -x0); pi: (-x0, -x1)
        want = {0: (x0[t], x1[t]), 1: (x1[t], -x0[t]), 2: (-x0[t], -x1[t]), 3: (-x1[t], x0[t])}[p]
        assert np.array_equal(y[t][..., 0::2], want[0]) and np.array_equal(y[t][..., 1::2], want[1])


def test_pair_norm_is_preserved():
    r, o = _run(T=64, NH=4, D=32, seed=1)
    x = r.x.float().numpy().astype(np.float64)
    y = o["y"].astype(np.float64)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-5, atol=1e-9)


def test_one_scale_per_head_matches_torch_cast():
    r, o = _run(T=50, NH=5, D=16, seed=2)
    y = torch.from_numpy(o["y"])
    for h in range(5):
        amax = y[:, h, :].abs().max().item()
        s = np.float32(amax) / np.float32(448.0)
        assert o["scales"][h] == s
        ref = (y[:, h, :] / torch.tensor(s)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(o["codes"][:, h, :], ref)


def test_scale_is_per_head_not_per_tensor():
    r = inputs.make_rope_inputs(20, 3, 16, 64, seed=4)
    x2 = r.x.clone()
    x2[:, 1, :] = (x2[:, 1, :].float() * 4).to(torch.bfloat16)  # exact: power of two
    a = oracle.inv_rope_quant(r.x, r.positions, r.cos, r.sin)
    b = oracle.inv_rope_quant(x2, r.positions, r.cos, r.sin)
    assert b["scales"][1] == 4 * a["scales"][1]
    assert b["scales"][0] == a["scales"][0] and b["scales"][2] == a["scales"][2]
    assert np.array_equal(a["codes"], b["codes"])


def test_zero_head_gets_scale_one():
    r = inputs.make_rope_inputs(4, 2, 8, 16, seed=5)
    x = r.x.clone()
    x[:, 0, :] = 0
    o = oracle.inv_rope_quant(x, r.positions, r.cos, r.sin)
    # all values zero (the sign of a zero product can give the code of -0)
    assert o["scales"][0] == 1.0 and not (o["codes"][:, 0, :] & 0x7F).any()


def test_rejects_bad_positions():
    r = inputs.make_rope_inputs(4, 2, 8, 16, seed=6)
    bad = r.positions.clone()
    bad[0] = 16
    try:
        oracle.inv_rope_quant(r.x, bad, r.cos, r.sin)
    except ValueError:
        return
    raise AssertionError("position outside the tables accepted")
