"""moe_quantize_e4m3_noalloc: the quantisation entry point for callers that
cannot allocate device memory (its scratch is a static device array of the
library).  Through the C ABI it must give exactly the codes and scale of
moe_quantize_e4m3, call after call, reusing the same array.

This file is collected last on purpose: it must pass in a fresh process (the
first call on the device looks up the array's address) and after every other
test has run."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_noalloc_matches_allocating_entry_point_on_consecutive_calls(gpu_lib):
    g = torch.Generator().manual_seed(1234)
    cases = [(64, 4096, 1.0), (7, 2048, 30.0)]  # two calls in a row, different sizes
    for T, H, amp in cases:
        x = (torch.randn(T, H, generator=g) * amp).to(torch.bfloat16).cuda()
        codes_ref, scale_ref = gpu_lib.moe_quantize_e4m3(x)
        codes, scale = gpu_lib.moe_quantize_e4m3_noalloc(x)
        torch.cuda.synchronize()
        # E4M3 codes are integers: bit-exact, like every quantisation test here
        assert np.array_equal(codes.cpu().numpy(), codes_ref.cpu().numpy())
        assert float(scale.item()) == float(scale_ref.item())
