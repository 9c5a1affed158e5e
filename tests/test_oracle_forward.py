"""Pins for the oracle's whole-layer forward.

The layer (English original page, Introduction and "Backend routing for FP8
tensor quantization"): token routing, data shuffling, expert computation, FP8
tensor scaling and expert aggregation in one pass.  The expert network is read
as a SwiGLU MLP (gate rows first, then up rows of w13; w2 down projection).

Pins, each independent of the oracle's own code:
  * E = 1, k = 1 reduces to a textbook SwiGLU MLP (torch fp64 matmul + silu);
  * k = E without renormalisation is the dense softmax-weighted mixture of all
    experts (torch fp64, scipy softmax);
  * permuting tokens permutes the output rows and routing exactly;
  * FP8: E = 1, k = 1 reduces to the SwiGLU MLP on tensors put through torch's
    own float8_e4m3fn cast with amax/448 scales; and the FP8 result stays within
    the E4M3 error bound of the unquantised result;
  * asking for a subset of output rows returns exactly those rows.
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from mixture_experts_layer_align_gb300 import inputs


def swiglu_ref(x, w13, w2):
    """Textbook SwiGLU MLP in fp64: W2 (silu(Wg x) * (Wu x))."""
    I = w13.shape[0] // 2
    g = x @ w13[:I].T
    u = x @ w13[I:].T
    return (torch.nn.functional.silu(g) * u) @ w2.T


def f64(t):
    return t.to(torch.float64)


def make(T, H, I, E, dtype, seed=0, routing="uniform"):
    w = inputs.make_weights(H, I, E, dtype, seed=seed)
    a = inputs.make_activations(T, H, E, routing, seed=seed)
    return w, a


def dequant(codes, scale):
    return codes.view(torch.float8_e4m3fn).to(torch.float64) * float(scale)


def torch_q(v64, s):
    """Quantise with torch's E4M3 cast (RNE), clamped first (satfinite)."""
    q = (v64.to(torch.float32) / torch.tensor(s, dtype=torch.float32)).clamp(-448, 448)
    return q.to(torch.float8_e4m3fn).to(torch.float64) * float(s)


def amax_scale(v):
    a = v.abs().max().to(torch.float32)
    return float(a / torch.tensor(448.0, dtype=torch.float32)) if a > 0 else 1.0


@pytest.mark.parametrize("renorm", [True, False])
def test_single_expert_bf16_is_swiglu(renorm):
    w, a = make(T=5, H=64, I=96, E=1, dtype="bf16")
    r = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, None, None, 1, renorm)
    ref = swiglu_ref(f64(a.x), f64(w.w13[0]), f64(w.w2[0])).numpy()
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-15)
    assert np.all(r["weights"] == 1.0)


def test_dense_mixture_bf16():
    T, H, I, E = 6, 32, 64, 5
    w, a = make(T, H, I, E, "bf16", seed=3)
    r = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, None, None, E, False)
    p = softmax(a.logits.numpy().astype(np.float64), axis=1)
    ref = np.zeros((T, H))
    for e in range(E):
        ref += p[:, e:e + 1] * swiglu_ref(f64(a.x), f64(w.w13[e]), f64(w.w2[e])).numpy()
    assert np.allclose(r["out"], ref, rtol=1e-11, atol=1e-14)


def test_sparse_mixture_bf16_by_library_routines():
    """k < E with renormalisation, checked against stable argsort + scipy
    softmax + torch fp64 SwiGLU per selected expert."""
    T, H, I, E, k = 7, 32, 64, 6, 2
    w, a = make(T, H, I, E, "bf16", seed=4)
    r = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, None, None, k, True)
    lg = a.logits.numpy()
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    p = np.take_along_axis(softmax(lg.astype(np.float64), axis=1), ids, 1)
    p = p / p.sum(1, keepdims=True)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            ref[t] += p[t, j] * swiglu_ref(f64(a.x[t:t + 1]), f64(w.w13[e]), f64(w.w2[e])).numpy()[0]
    assert np.array_equal(r["ids"], ids)
    assert np.allclose(r["out"], ref, rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_token_permutation_invariance(dtype):
    T, H, I, E, k = 9, 128, 128, 8, 3
    w, a = make(T, H, I, E, dtype, seed=5)
    s13, s2 = w.w13_scale, w.w2_scale
    r = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, s13, s2, k, True)
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(1))
    r2 = oracle.moe_forward(a.x[perm], a.logits[perm], w.w13, w.w2, s13, s2, k, True)
    assert np.array_equal(r2["ids"], r["ids"][perm.numpy()])
    assert np.array_equal(r2["out"], r["out"][perm.numpy()])


def test_single_expert_fp8_is_swiglu_on_quantised_tensors():
    T, H, I = 6, 128, 256
    w, a = make(T, H, I, 1, "fp8", seed=6)
    r = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, 1, True)
    x = f64(a.x)
    sx = amax_scale(x)
    xq = torch_q(x, sx)
    w13 = dequant(w.w13[0], w.w13_scale[0])
    w2 = dequant(w.w2[0], w.w2_scale[0])
    g, u = xq @ w13[:I].T, xq @ w13[I:].T
    h = torch.nn.functional.silu(g) * u
    sh = amax_scale(h)
    ref = (torch_q(h, sh) @ w2.T).numpy()
    assert r["s_x"] == pytest.approx(sx, rel=0, abs=0)
    assert r["s_h"] == pytest.approx(sh, rel=1e-6)
    # an h value sitting on a rounding boundary may quantise to a neighbour
    # code when the two fp64 accumulation orders differ in the last bit
    err = np.abs(r["out"] - ref).max() / np.abs(ref).max()
    assert err < 1e-6, err


def test_dense_mixture_fp8():
    """k = E, no renormalisation: sum_e p_e * W2_e q(h_e) with one s_h over all
    pairs, built from torch's cast."""
    T, H, I, E = 4, 128, 128, 4
    w, a = make(T, H, I, E, "fp8", seed=7)
    r = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, E, False)
    p = softmax(a.logits.numpy().astype(np.float64), axis=1)
    xq = torch_q(f64(a.x), amax_scale(f64(a.x)))
    hs = []
    for e in range(E):
        w13 = dequant(w.w13[e], w.w13_scale[e])
        hs.append(torch.nn.functional.silu(xq @ w13[:I].T) * (xq @ w13[I:].T))
    sh = amax_scale(torch.stack(hs))
    ref = np.zeros((T, H))
    for e in range(E):
        ref += p[:, e:e + 1] * (torch_q(hs[e], sh) @ dequant(w.w2[e], w.w2_scale[e]).T).numpy()
    err = np.abs(r["out"] - ref).max() / np.abs(ref).max()
    assert err < 1e-6, err


def test_fp8_within_e4m3_error_of_unquantised():
    """Same codes/scales for the weights; the only differences are the two
    activation quantisations (relative step 2^-4 for normal E4M3 values), so
    the result must stay within a few percent of the unquantised layer."""
    T, H, I, E, k = 16, 256, 256, 8, 2
    w, a = make(T, H, I, E, "fp8", seed=8)
    r = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
    ids, wt = r["ids"], r["weights"]
    x = f64(a.x)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            w13 = dequant(w.w13[e], w.w13_scale[e])
            w2 = dequant(w.w2[e], w.w2_scale[e])
            ref[t] += wt[t, j] * swiglu_ref(x[t:t + 1], w13, w2).numpy()[0]
    err = np.abs(r["out"] - ref).max() / np.abs(ref).max()
    assert 1e-4 < err < 0.1, err   # quantisation is visible, but bounded


def test_row_subset_equals_full():
    T, H, I, E, k = 10, 128, 128, 8, 2
    for dtype in ("bf16", "fp8"):
        w, a = make(T, H, I, E, dtype, seed=9)
        full = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
        rows = [7, 0, 3]
        sub = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True,
                                 rows=rows)
        assert np.array_equal(sub["out"], full["out"][rows])


def test_zero_input_gives_zero_and_unit_scales():
    T, H, I, E, k = 3, 128, 128, 4, 2
    w, a = make(T, H, I, E, "fp8", seed=10)
    x = torch.zeros_like(a.x)
    r = oracle.moe_forward(x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
    assert np.all(r["out"] == 0) and r["s_x"] == 1.0 and r["s_h"] == 1.0
