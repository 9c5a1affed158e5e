"""moe_quantize_e4m3_noalloc: the activation quantisation entry point for
callers that cannot allocate device memory where they call it (another
component owns every allocation, or the thread must not take cudaMalloc's
implicit synchronisation).  Its scratch is a static device array of the
library, so the caller passes only inputs and outputs.

Through the C ABI, on two calls in a row, it must give exactly the codes and
scale of the allocating entry point moe_quantize_e4m3 and of the CPU oracle,
including a tensor large enough to use the most partial maxima the entry
point ever takes.  One test runs in this process (after every other test
file: pytest collects this file last); another runs the same check in a fresh
Python process whose first CUDA work is the no-alloc call, so that the
first-call lookup of the array's address is exercised there.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (T, H, amplitude): the last one has T*H / 8 / 256 = 8192 amax CTAs of
# work, so the entry point takes its largest partial count (4 per SM).
CASES = [(64, 4096, 1.0), (7, 2048, 30.0), (8192, 2048, 3.0)]


def _check_case(moe, T, H, amp, seed):
    g = torch.Generator().manual_seed(seed)
    x_cpu = (torch.randn(T, H, generator=g) * amp).to(torch.bfloat16)
    x = x_cpu.cuda()
    codes, scale = moe.moe_quantize_e4m3_noalloc(x)
    codes_ref, scale_ref = moe.moe_quantize_e4m3(x)
    torch.cuda.synchronize()
    got = codes.cpu().numpy()
    # E4M3 codes are integers: bit-exact against both references
    assert np.array_equal(got, codes_ref.cpu().numpy())
    assert float(scale.item()) == float(scale_ref.item())
    o_codes, o_scale = oracle.quantize_act(x_cpu)
    assert float(scale.item()) == o_scale
    assert np.array_equal(got, o_codes)


def test_noalloc_matches_allocating_entry_point_and_oracle_on_consecutive_calls(gpu_lib):
    for i, (T, H, amp) in enumerate(CASES):
        _check_case(gpu_lib, T, H, amp, 1234 + i)


_FRESH = r"""
import sys
sys.path.insert(0, {root!r})
import torch
import mixture_experts_layer_align_gb300 as moe
sys.path.insert(0, {tests!r})
from test_zz_no_alloc import CASES, _check_case
moe.load()
torch.cuda.set_device(0)
for i, (T, H, amp) in enumerate(CASES):
    _check_case(moe, T, H, amp, 99 + i)
print("fresh-process no-alloc calls ok")
"""


def test_noalloc_first_call_in_a_fresh_process(gpu_lib):
    code = _FRESH.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fresh-process no-alloc calls ok" in r.stdout
