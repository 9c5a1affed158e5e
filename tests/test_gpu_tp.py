"""Tensor-parallel shards of the layer on the GPU (the library's two-call
form), emulated rank by rank on one device: every rank's gate/up call, the
maximum of the ranks' max |h| words written back into every workspace (what
an all-reduce MAX does), every rank's down call, and the sum of the partial
outputs (what an all-reduce SUM does) must match the unsharded oracle within
the layer's tolerance; the unchanged single-GPU kernels run on each shard."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_out_close
from mixture_experts_layer_align_gb300 import inputs, tp

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,T,H,I,E,k,world", [
    ("fp8", 9, 256, 512, 8, 2, 2),
    ("fp8", 64, 512, 1024, 16, 4, 4),
    ("fp8", 300, 256, 512, 8, 2, 2),     # several row tiles per expert
    ("bf16", 5, 128, 256, 4, 2, 2),
])
def test_shards_sum_to_the_unsharded_layer(gpu_lib, dtype, T, H, I, E, k, world):
    moe = gpu_lib
    w = inputs.make_weights(H, I, E, dtype, seed=T, device="cuda")
    a = inputs.make_activations(T, H, E, "uniform", seed=T, device="cuda")
    fp8 = dtype == "fp8"
    dt = moe.MOE_DT_FP8_E4M3 if fp8 else moe.MOE_DT_BF16
    shards = [tp.shard_weights(w.w13, w.w2, r, world) for r in range(world)]
    wss = [moe.alloc_workspace(T, H, I // world, E, k, dt) for _ in range(world)]
    outs = [torch.empty(T, H, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
    for r in range(world):
        moe.moe_fused_forward_gate_up(a.x, a.logits, shards[r][0], shards[r][1], w.w13_scale,
                                      w.w2_scale, k, True, outs[r], wss[r])
    if fp8:
        amax = torch.stack([moe.h_amax_view(ws) for ws in wss]).max()
        for ws in wss:
            moe.h_amax_view(ws).copy_(amax)
    for r in range(world):
        moe.moe_fused_forward_down(a.x, a.logits, shards[r][0], shards[r][1], w.w13_scale,
                                   w.w2_scale, k, True, outs[r], wss[r])
    for ws in wss:
        assert moe.moe_check_status(ws) == 0
    total = torch.stack([o.float() for o in outs]).sum(0)
    ref = oracle.moe_forward(a.x.cpu(), a.logits.cpu(), w.w13.cpu(), w.w2.cpu(),
                             None if w.w13_scale is None else w.w13_scale.cpu(),
                             None if w.w2_scale is None else w.w2_scale.cpu(), k, True)
    assert_out_close(total, ref["out"])
    if fp8:
        # the max-reduced word is the unsharded max |h| (fp32 rounding of h on
        # the GPU against fp64 in the oracle)
        assert abs(float(amax.item()) - ref["h_amax"]) <= 1e-3 * ref["h_amax"]


def test_two_calls_equal_one_call_and_tp_forward_alone(gpu_lib):
    moe = gpu_lib
    T, H, I, E, k = 37, 256, 512, 8, 2
    w = inputs.make_weights(H, I, E, "fp8", seed=4, device="cuda")
    a = inputs.make_activations(T, H, E, "uniform", seed=4, device="cuda")
    one = moe.moe_fused_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
    alone = tp.tp_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
    torch.cuda.synchronize()
    d = (one.float() - alone.float()).abs().max().item()
    assert d <= 1e-2 * one.float().abs().max().item()
    assert np.isfinite(alone.float().cpu().numpy()).all()
