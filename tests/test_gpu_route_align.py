"""GPU parity: router, alignment by expert and activation quantisation through
the C ABI, against the CPU oracle (bit-exact on ids, counts, permutation and
E4M3 codes)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import W_ATOL, W_RTOL
from mixture_experts_layer_align_gb300 import inputs

pytestmark = pytest.mark.gpu


def _logits(T, E, kind, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(T, E, generator=g)
    if kind == "ties":
        vals = torch.tensor([-1.0, -0.0, 0.0, 0.5, 1.0, 2.0])
        return vals[torch.randint(0, len(vals), (T, E), generator=g)]
    if kind == "zipf":
        return torch.randn(T, E, generator=g) + inputs.zipf_bias(E)
    if kind == "large":
        return torch.randn(T, E, generator=g) * 1e4
    raise ValueError(kind)


@pytest.mark.parametrize("T,E,k,kind", [
    (1, 8, 2, "normal"), (4, 8, 2, "ties"), (37, 128, 8, "normal"), (513, 256, 8, "zipf"),
    (64, 1, 1, "normal"), (100, 16, 16, "ties"), (300, 1024, 8, "normal"), (200, 64, 40, "large"),
    (8192, 128, 8, "normal"),
])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_topk_parity(gpu_lib, T, E, k, kind, renorm):
    lg = _logits(T, E, kind, seed=T * 7 + E).contiguous()
    ids, w = gpu_lib.moe_route_topk(lg.cuda(), k, renorm)
    torch.cuda.synchronize()
    ref_ids, ref_w = oracle.route_topk(lg, k, renorm)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=W_RTOL, atol=W_ATOL)


# More router cases drawn once with random.Random(31): E 1..1024, k up to 32,
# T up to 5000, every logit kind (ties, Zipf bias, |logits| ~ 1e4).
@pytest.mark.parametrize("T,E,k,kind", [
    (5, 1, 1, "large"), (1, 7, 6, "ties"), (31, 2, 1, "ties"), (1, 1024, 3, "ties"),
    (5000, 31, 18, "large"), (5, 31, 19, "normal"), (1000, 1, 1, "ties"), (4096, 31, 11, "zipf"),
    (64, 257, 16, "ties"), (1, 100, 4, "ties"), (64, 33, 9, "ties"), (5, 100, 2, "large"),
])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_topk_random_cases(gpu_lib, T, E, k, kind, renorm):
    test_route_topk_parity(gpu_lib, T, E, k, kind, renorm)


def test_route_zero_tokens(gpu_lib):
    lg = torch.zeros(0, 8, device="cuda")
    ids, w = gpu_lib.moe_route_topk(lg, 2, True)
    assert ids.shape == (0, 2)


@pytest.mark.parametrize("T,k,E,bm,kind", [
    (4, 2, 8, 16, "normal"), (1, 8, 128, 16, "normal"), (256, 8, 128, 16, "normal"),
    (128, 8, 256, 16, "zipf"), (1000, 3, 5, 1, "normal"), (2048, 8, 128, 64, "zipf"),
    (8192, 8, 128, 16, "normal"), (8192, 8, 128, 128, "zipf"), (3000, 8, 1024, 7, "normal"),
    (5, 1, 1, 256, "normal"),
])
def test_align_parity(gpu_lib, T, k, E, bm, kind):
    lg = _logits(T, E, kind, seed=T + k + E)
    ref_ids, _ = oracle.route_topk(lg, k, True)
    ids = torch.from_numpy(ref_ids).cuda()
    res = gpu_lib.moe_align_by_expert(ids, E, bm)
    torch.cuda.synchronize()
    ref = oracle.align(ref_ids, E, bm)
    n = ref["num_padded"]
    assert int(res["num_padded"].item()) == n
    assert np.array_equal(res["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(res["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(res["sorted_ids"][:n].cpu().numpy(), ref["sorted_ids"])
    assert np.array_equal(res["tile_expert"][:n // bm].cpu().numpy(), ref["tile_expert"])
    # entries past the padded end are not written
    assert torch.all(res["sorted_ids"][n:] == -1)


# More alignment cases drawn once with random.Random(31): E 1..1024, k up to 8,
# T up to 7000 (up to 49,000 pairs), block_m from 1 to 256.
@pytest.mark.parametrize("T,k,E,bm,kind", [
    (7000, 4, 64, 33, "zipf"), (100, 4, 256, 128, "normal"), (100, 1, 1024, 16, "ties"),
    (600, 7, 256, 128, "zipf"), (4100, 4, 256, 1, "ties"), (1, 5, 8, 2, "normal"),
    (4100, 1, 1, 1, "zipf"), (100, 5, 513, 128, "normal"), (9, 2, 3, 256, "ties"),
    (7000, 7, 1024, 1, "zipf"), (1, 2, 3, 256, "zipf"), (9, 1, 3, 16, "normal"),
])
def test_align_random_cases(gpu_lib, T, k, E, bm, kind):
    test_align_parity(gpu_lib, T, k, E, bm, kind)


def test_align_out_of_range_ids_are_skipped(gpu_lib):
    ids = torch.tensor([[0, 5], [9, 1], [-1, 1]], dtype=torch.int32, device="cuda")
    res = gpu_lib.moe_align_by_expert(ids, 6, 4)
    torch.cuda.synchronize()
    assert res["counts"].cpu().tolist() == [1, 2, 0, 0, 0, 1]
    assert res["sorted_ids"][:12].cpu().tolist() == [0, 6, 6, 6, 3, 5, 6, 6, 1, 6, 6, 6]


@pytest.mark.parametrize("T,H,scale", [(1, 4096, 1.0), (64, 4096, 1.0), (8192, 2048, 1.0),
                                       (7, 7168, 1e-3), (3, 128, 0.0), (5, 256, 300.0)])
def test_quantize_e4m3_bit_exact(gpu_lib, T, H, scale):
    g = torch.Generator().manual_seed(T + H)
    x = (torch.randn(T, H, generator=g) * scale).to(torch.bfloat16)
    if T > 3:
        x[0, 0] = 0.0  # exact zero
        x[1, 1] = -x[1, 1]
    codes, s = gpu_lib.moe_quantize_e4m3(x.cuda())
    torch.cuda.synchronize()
    ref_codes, ref_s = oracle.quantize_act(x)
    assert float(s.item()) == ref_s
    assert np.array_equal(codes.cpu().numpy(), ref_codes)


@pytest.mark.parametrize("amax_bits", [0x43E0, 0x43E2, 0x3F81, 0x4011, 0x3A83, 0x4C35])
def test_quantize_e4m3_every_bf16_value(gpu_lib, amax_bits):
    """Every finite bf16 value of magnitude <= amax, both signs, under the scale
    amax / 448: the kernels' codes from two bracketing products (division only
    where those disagree) must be the code of the correctly rounded quotient
    for each of them, including the values whose quotient falls near an E4M3
    rounding midpoint."""
    amax = np.array([amax_bits], np.uint16).view(np.uint16)[0]
    pos = np.arange(0, 0x7F80, dtype=np.uint16)          # +0 .. largest finite
    pos = pos[pos <= amax]
    vals = np.concatenate([pos, pos | np.uint16(0x8000)])
    vals = np.concatenate([vals, np.full((-vals.size) % 128, 0, np.uint16)])
    x = torch.from_numpy(vals.view(np.int16).copy()).view(torch.bfloat16).reshape(-1, 128)
    codes, s = gpu_lib.moe_quantize_e4m3(x.cuda())
    torch.cuda.synchronize()
    ref_codes, ref_s = oracle.quantize_act(x)
    assert float(s.item()) == ref_s
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
