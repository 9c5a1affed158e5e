"""Bounded device waits: a forced wait on a barrier nothing arrives on must end
with MOE_ERR_DEVICE_TIMEOUT reported through the workspace status word, and
the CUDA context must stay usable for the next call (no trap, no fault)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_out_close
from mixture_experts_layer_align_gb300 import inputs

pytestmark = pytest.mark.gpu


# Small batches: the kernel sequence and, with MOE_FLAG_ONE_KERNEL (0x20),
# the single cooperative kernel (its CTAs also wait on grid-wide counters):
# (8, ...) decode-style tiles (I = 2176 > 2048 keeps the down weights in M);
# (600, ...) 300 rows per expert: wide gate/up tiles on one SM each (I = 128),
# tokens in M for down.  (1200, ...) wide gate/up tiles on SM pairs;
# (4096, ...) the same, with the down GEMM combining through bf16 rows (TMA
# stores) and the row-combine kernel.
@pytest.mark.parametrize("T,H,I,E,k,flags", [
    (8, 256, 256, 8, 2, 0), (8, 256, 2176, 4, 2, 0), (600, 256, 128, 4, 2, 0),
    (8, 256, 256, 8, 2, 0x20), (8, 256, 2176, 4, 2, 0x20), (600, 256, 128, 4, 2, 0x20),
    (1200, 256, 512, 4, 2, 0), (4096, 1024, 256, 4, 2, 0)])
def test_forced_timeout_reports_status_and_context_survives(gpu_lib, T, H, I, E, k, flags):
    assert flags in (0, gpu_lib.MOE_FLAG_ONE_KERNEL)
    w = inputs.make_weights(H, I, E, "fp8", seed=11)
    a = inputs.make_activations(T, H, E, "uniform", seed=11)
    d = dict(x=a.x.cuda(), lg=a.logits.cuda(), w13=w.w13.cuda(), w2=w.w2.cuda(),
             s13=w.w13_scale.cuda(), s2=w.w2_scale.cuda())
    ws = gpu_lib.alloc_workspace(T, H, I, E, k, gpu_lib.MOE_DT_FP8_E4M3)
    gpu_lib.moe_fused_forward(d["x"], d["lg"], d["w13"], d["w2"], d["s13"], d["s2"], k, True,
                              workspace=ws, debug_flags=gpu_lib.MOE_DEBUG_FORCE_TIMEOUT | flags)
    assert gpu_lib.moe_check_status(ws) == 5  # MOE_ERR_DEVICE_TIMEOUT
    # the context is intact: a normal call on the same workspace is correct
    out = gpu_lib.moe_fused_forward(d["x"], d["lg"], d["w13"], d["w2"], d["s13"], d["s2"], k,
                                    True, workspace=ws, debug_flags=flags)
    assert gpu_lib.moe_check_status(ws) == 0
    ref = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
    assert_out_close(out, ref["out"])
    assert torch.cuda.is_available()
    assert np.isfinite(out.float().cpu().numpy()).all()
