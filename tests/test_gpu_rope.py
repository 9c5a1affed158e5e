"""GPU parity of the inverse rotary embedding + per-head FP8 quantisation
against the CPU oracle: codes and scales bit-exact (both sides round the same
fp32 products and sums and divide in IEEE fp32), at shapes with ragged token
counts, every supported head size, and a position outside the tables."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_align_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,NH,D,max_pos", [
    (1, 1, 8, 4), (37, 6, 64, 512), (257, 8, 128, 4096), (1000, 3, 256, 2048),
    (129, 5, 16, 64), (4096, 32, 128, 8192), (8192, 8, 32, 8192),
    (20000, 3, 256, 2048),   # two launches, one head vector per warp iteration
    (12000, 40, 16, 64),     # two launches, a partial group of heads
    (2000, 1024, 8, 64),     # two launches, 32 head vectors of 8 per warp iteration
])
def test_inv_rope_quant_matches_oracle(gpu_lib, T, NH, D, max_pos):
    r = inputs.make_rope_inputs(T, NH, D, max_pos, seed=T)
    ref = oracle.inv_rope_quant(r.x, r.positions, r.cos, r.sin)
    codes, scales, scratch = gpu_lib.moe_inv_rope_quant_per_head(
        r.x.cuda(), r.positions.cuda(), r.cos.cuda(), r.sin.cuda())
    assert gpu_lib.moe_check_status(scratch) == 0
    assert np.array_equal(scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(codes.cpu().numpy(), ref["codes"])


# More shapes drawn once with random.Random(47): head sizes 8..256, 1..512 heads,
# T up to 9000, tables of 1..8192 positions (max_pos = 1: every position is 0).
@pytest.mark.parametrize("T,NH,D,max_pos", [
    (300, 2, 32, 8192), (17, 33, 64, 8192), (1217, 100, 64, 1), (1, 1, 64, 1),
    (1217, 33, 8, 1000), (1217, 7, 16, 8192), (2, 512, 32, 1), (3000, 33, 128, 64),
    (1217, 33, 128, 8192), (9000, 7, 16, 1),
])
def test_inv_rope_quant_random_shapes(gpu_lib, T, NH, D, max_pos):
    test_inv_rope_quant_matches_oracle(gpu_lib, T, NH, D, max_pos)


def test_zero_head_and_repeat_calls(gpu_lib):
    r = inputs.make_rope_inputs(64, 4, 64, 128, seed=9)
    x = r.x.clone()
    x[:, 2, :] = 0
    ref = oracle.inv_rope_quant(x, r.positions, r.cos, r.sin)
    args = (x.cuda(), r.positions.cuda(), r.cos.cuda(), r.sin.cuda())
    for _ in range(2):  # the scratch and outputs of a previous call do not leak in
        codes, scales, scratch = gpu_lib.moe_inv_rope_quant_per_head(*args)
        assert np.array_equal(scales.cpu().numpy(), ref["scales"])
        assert np.array_equal(codes.cpu().numpy(), ref["codes"])


def test_position_outside_tables_is_reported(gpu_lib):
    r = inputs.make_rope_inputs(16, 2, 32, 64, seed=10)
    pos = r.positions.clone()
    pos[3] = 64  # one past the tables: read as position 0, status word set
    codes, scales, scratch = gpu_lib.moe_inv_rope_quant_per_head(
        r.x.cuda(), pos.cuda(), r.cos.cuda(), r.sin.cuda())
    assert gpu_lib.moe_check_status(scratch) == 6  # MOE_ERR_DEVICE_RANGE
    pos[3] = 0
    ref = oracle.inv_rope_quant(r.x, pos, r.cos, r.sin)
    assert np.array_equal(codes.cpu().numpy(), ref["codes"])
    # the next good call clears the status
    _, _, scratch = gpu_lib.moe_inv_rope_quant_per_head(
        r.x.cuda(), pos.cuda(), r.cos.cuda(), r.sin.cuda(), scratch=scratch)
    assert gpu_lib.moe_check_status(scratch) == 0


def test_position_outside_tables_large_input(gpu_lib):
    """The two-launch path (per-head words by atomic max, flag word after
    them) reports a bad position and clears the status on the next call."""
    r = inputs.make_rope_inputs(4096, 32, 128, 8192, seed=12)
    pos = r.positions.clone()
    pos[1000] = -1
    codes, scales, scratch = gpu_lib.moe_inv_rope_quant_per_head(
        r.x.cuda(), pos.cuda(), r.cos.cuda(), r.sin.cuda())
    assert gpu_lib.moe_check_status(scratch) == 6  # MOE_ERR_DEVICE_RANGE
    pos[1000] = 0
    ref = oracle.inv_rope_quant(r.x, pos, r.cos, r.sin)
    assert np.array_equal(scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(codes.cpu().numpy(), ref["codes"])
    _, _, scratch = gpu_lib.moe_inv_rope_quant_per_head(
        r.x.cuda(), pos.cuda(), r.cos.cuda(), r.sin.cuda(), scratch=scratch)
    assert gpu_lib.moe_check_status(scratch) == 0


@pytest.mark.parametrize("T", [64, 4096])  # one cooperative launch; memset + two launches
def test_graph_replay_equals_eager(gpu_lib, T):
    """Captured once in a CUDA graph and replayed on new inputs written into
    the same buffers, the operation gives the eager (and oracle) result."""
    NH, D, max_pos = 32, 128, 8192
    a = inputs.make_rope_inputs(T, NH, D, max_pos, seed=T)
    b = inputs.make_rope_inputs(T, NH, D, max_pos, seed=T + 1)
    x, pos = a.x.cuda(), a.positions.cuda()
    cos_t, sin_t = a.cos.cuda(), a.sin.cuda()
    codes = torch.empty(T, NH, D, dtype=torch.uint8, device="cuda")
    scales = torch.empty(NH, dtype=torch.float32, device="cuda")
    scratch = torch.empty(gpu_lib.moe_inv_rope_scratch_size(T, NH, D), dtype=torch.uint8,
                          device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gpu_lib.moe_inv_rope_quant_per_head(x, pos, cos_t, sin_t, codes, scales, scratch)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu_lib.moe_inv_rope_quant_per_head(x, pos, cos_t, sin_t, codes, scales, scratch)
    x.copy_(b.x.cuda())
    pos.copy_(b.positions.cuda())
    graph.replay()
    torch.cuda.synchronize()
    assert gpu_lib.moe_check_status(scratch) == 0
    ref = oracle.inv_rope_quant(b.x, b.positions, a.cos, a.sin)
    assert np.array_equal(scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(codes.cpu().numpy(), ref["codes"])


def _boundary_values(amax):
    """fp32 values y whose quotients y / s (s = amax / 448, IEEE fp32) sit on
    and around every E4M3 rounding boundary (the midpoints between consecutive
    codes, subnormal ones included) and every E4M3 value, 6 ulps either side,
    both signs; amax itself first, so that it is the head's maximum."""
    c = np.arange(127)
    e, m = c >> 3, c & 7
    vals = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8) * 2.0 ** (e - 7))
    mids = (vals[:-1] + vals[1:]) / 2
    s = np.float32(amax) / np.float32(448)
    ys = []
    for t in np.concatenate([mids, vals[1:]]):
        y0 = np.array([np.float64(t) * np.float64(s)], np.float32)
        for k in range(-6, 7):
            y = (y0.view(np.int32) + k).view(np.float32)[0]
            if 0 < y < amax:
                ys += [y, -y]
    return np.array([np.float32(amax)] + ys, np.float32)


@pytest.mark.parametrize("T", [None, 12000])
def test_inv_rope_quant_codes_at_e4m3_boundaries(gpu_lib, T):
    # x pairs (1, 0) in head 0 and (0, 1) in head 1 turn the rotation into
    # y = (c, -s) and (s, c): the caller's tables place y anywhere in fp32.
    # T = None: one cooperative launch; 12000 tokens: the two-launch path.
    amax = np.float32(3.7)
    ys = _boundary_values(amax)
    n = -(-ys.size // 8)
    rng = np.random.default_rng(3)
    pad = rng.uniform(-amax, amax, n * 8 - ys.size).astype(np.float32)
    ys = np.concatenate([ys, pad]).reshape(n, 4, 2)
    T = n if T is None else T
    reps = -(-T // n)
    cos = np.tile(ys[:, :, 0], (reps, 1))[:T]
    sin = -np.tile(ys[:, :, 1], (reps, 1))[:T]
    x = torch.zeros(T, 2, 8, dtype=torch.bfloat16)
    x[:, 0, 0::2] = 1
    x[:, 1, 1::2] = 1
    pos = torch.arange(T, dtype=torch.int32)
    cos_t, sin_t = torch.from_numpy(np.ascontiguousarray(cos)), torch.from_numpy(np.ascontiguousarray(sin))
    ref = oracle.inv_rope_quant(x, pos, cos_t, sin_t)
    assert ref["scales"][0] == np.float32(amax) / np.float32(448)
    codes, scales, scratch = gpu_lib.moe_inv_rope_quant_per_head(
        x.cuda(), pos.cuda(), cos_t.cuda(), sin_t.cuda())
    assert gpu_lib.moe_check_status(scratch) == 0
    assert np.array_equal(scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(codes.cpu().numpy(), ref["codes"])
