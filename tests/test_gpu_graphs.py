"""Shape genericity of the fused forward: CUDA-graph capture and first calls.

Every shape is a runtime argument of the same kernels: the library compiles
nothing and builds no per-shape plan at call time.  So (1) a call can be
captured into a CUDA graph and replayed on new inputs written into the
captured buffers, matching an eager call on those inputs, and (2) the first
call at a token count the process has not seen costs about what the next
calls at that count cost (no JIT, no plan building).
"""
import statistics
import time

import pytest
import torch

from mixture_experts_layer_align_gb300 import inputs

pytestmark = pytest.mark.gpu

H, I, E, K = 2048, 768, 128, 8   # fine-grained / prefill expert shape
TMAX = 6144


@pytest.fixture(scope="module")
def setup(gpu_lib):
    moe = gpu_lib
    w = inputs.make_weights(H, I, E, "fp8", seed=0, device="cuda")
    a = inputs.make_activations(TMAX, H, E, "uniform", seed=0, device="cuda")
    ws = moe.alloc_workspace(TMAX, H, I, E, K, moe.MOE_DT_FP8_E4M3, "cuda")
    return moe, w, a, ws


def _call(moe, w, ws, x, lg, out):
    moe.moe_fused_forward(x, lg, w.w13, w.w2, w.w13_scale, w.w2_scale, K, True, out=out,
                          workspace=ws)


@pytest.mark.parametrize("T", [1, 37, 512, 2600])
def test_graph_capture_replays_on_new_inputs(setup, T):
    moe, w, a, ws = setup
    gx = a.x[:T].clone()
    gl = a.logits[:T].clone()
    go = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _call(moe, w, ws, gx, gl, go)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _call(moe, w, ws, gx, gl, go)
    for seed in (T + 1, T + 2):
        fresh = inputs.make_activations(T, H, E, "uniform", seed=seed, device="cuda")
        gx.copy_(fresh.x)
        gl.copy_(fresh.logits)
        g.replay()
        ref = torch.empty_like(go)
        _call(moe, w, ws, fresh.x, fresh.logits, ref)
        torch.cuda.synchronize()
        assert moe.moe_check_status(ws) == 0
        scale = ref.float().abs().max().item()
        assert scale > 0
        # same kernels, same inputs: only the fp32 summation order of the combine differs
        assert (go.float() - ref.float()).abs().max().item() <= 1e-2 * scale


def test_first_call_at_a_new_token_count_costs_a_steady_call(setup):
    moe, w, a, ws = setup
    out = torch.empty(TMAX, H, dtype=torch.bfloat16, device="cuda")
    _call(moe, w, ws, a.x[:5], a.logits[:5], out[:5])  # library set-up happens here
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    prev = 5
    for T in (3, 11, 29, 77, 131, 257, 513, 1031, 2049, 3001, 4099, 6007):
        x, lg, o = a.x[:T], a.logits[:T], out[:T]
        # the GPU is busy with an earlier call while the first one is enqueued
        _call(moe, w, ws, a.x[:prev], a.logits[:prev], out[:prev])
        prev = T
        h0 = time.perf_counter()
        ev[0].record()
        _call(moe, w, ws, x, lg, o)
        ev[1].record()
        host_us = (time.perf_counter() - h0) * 1e6
        for i in range(3):
            _call(moe, w, ws, x, lg, o)
            ev[2 + i].record()
        torch.cuda.synchronize()
        first = ev[0].elapsed_time(ev[1]) * 1e3
        steady = statistics.median(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(1, 4))
        # a per-shape compile or plan would cost milliseconds of host time
        assert host_us < 5000, (T, host_us)
        assert first <= 2.0 * steady + 50.0, (T, first, steady)
    assert moe.moe_check_status(ws) == 0
