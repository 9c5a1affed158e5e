"""Concurrent calls: the library keeps no per-call state outside the caller's
workspace, so calls on different streams (each with its own workspace) may
overlap, and host threads may enqueue calls at the same time.  Every result
must equal the oracle's."""
import threading

import pytest
import torch

import oracle
from helpers import assert_out_close
from mixture_experts_layer_align_gb300 import inputs

pytestmark = pytest.mark.gpu

SHAPES = [(16, 256, 512, 8, 2), (300, 256, 512, 16, 4), (5000, 256, 256, 8, 2)]


def _case(i, T, H, I, E, k):
    w = inputs.make_weights(H, I, E, "fp8", seed=100 + i)
    a = inputs.make_activations(T, H, E, "zipf" if i % 2 else "uniform", seed=100 + i)
    ref = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
    dev = dict(x=a.x.cuda(), lg=a.logits.cuda(), w13=w.w13.cuda(), w2=w.w2.cuda(),
               s13=w.w13_scale.cuda(), s2=w.w2_scale.cuda())
    return (T, H, I, E, k), dev, ref["out"]


def test_calls_on_separate_streams_overlap_correctly(gpu_lib):
    cases = [_case(i, *s) for i, s in enumerate(SHAPES)]
    streams = [torch.cuda.Stream() for _ in cases]
    wss, outs = [], []
    for (T, H, I, E, k), d, _ in cases:
        wss.append(gpu_lib.alloc_workspace(T, H, I, E, k, gpu_lib.MOE_DT_FP8_E4M3))
        outs.append(torch.empty(T, H, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    for _ in range(3):  # interleaved launches on the three streams
        for (shape, d, _), st, ws, out in zip(cases, streams, wss, outs):
            with torch.cuda.stream(st):
                gpu_lib.moe_fused_forward(d["x"], d["lg"], d["w13"], d["w2"], d["s13"], d["s2"],
                                          shape[4], True, out=out, workspace=ws)
    torch.cuda.synchronize()
    for (shape, d, ref), ws, out in zip(cases, wss, outs):
        assert gpu_lib.moe_check_status(ws) == 0
        assert_out_close(out, ref)


def test_calls_from_several_host_threads(gpu_lib):
    cases = [_case(i, *s) for i, s in enumerate(SHAPES)]
    results, errors = [None] * len(cases), []

    def run(j):
        try:
            (T, H, I, E, k), d, _ = cases[j]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                ws = gpu_lib.alloc_workspace(T, H, I, E, k, gpu_lib.MOE_DT_FP8_E4M3)
                for _ in range(3):
                    out = gpu_lib.moe_fused_forward(d["x"], d["lg"], d["w13"], d["w2"], d["s13"],
                                                    d["s2"], k, True, workspace=ws)
            st.synchronize()
            results[j] = (out, gpu_lib.moe_check_status(ws, st))
        except Exception as e:  # reported below, on the test's thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(j,)) for j in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (_, _, ref), (out, status) in zip(cases, results):
        assert status == 0
        assert_out_close(out, ref)
