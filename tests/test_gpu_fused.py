"""GPU parity of the fused MoE forward against the CPU oracle.

Routing (expert ids, per-expert counts) must match bit-exactly; outputs within
max|gpu - oracle| <= 2e-2 * max|oracle|.  Small cases and the five measured
workloads at full size are compared on every output element; 8192-token
prefill on 512 rows that cover every expert's segment (every row under
`-m slow`).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import W_ATOL, W_RTOL, assert_out_close
from mixture_experts_layer_align_gb300 import inputs

pytestmark = pytest.mark.gpu


def run_case(moe, w, a, top_k, renorm, rows=None, repeat=1, flags=0):
    dev = "cuda"
    T, E = a.T, w.E
    x, lg = a.x.to(dev), a.logits.to(dev)
    w13, w2 = w.w13.to(dev), w.w2.to(dev)
    s13 = None if w.w13_scale is None else w.w13_scale.to(dev)
    s2 = None if w.w2_scale is None else w.w2_scale.to(dev)
    ids = torch.empty(T, top_k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, top_k, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    ws = moe.alloc_workspace(T, w.H, w.I, E, top_k, 1 if s13 is not None else 0, dev)
    ws.fill_(0xAB)  # the call must not rely on a zeroed workspace
    for _ in range(repeat):
        out = moe.moe_fused_forward(x, lg, w13, w2, s13, s2, top_k, renorm, workspace=ws,
                                    topk_ids_out=ids, topk_w_out=wts, counts_out=counts,
                                    debug_flags=flags)
    assert moe.moe_check_status(ws) == 0
    ref = oracle.moe_forward(a.x, a.logits, w.w13.cpu(), w.w2.cpu(),
                             None if w.w13_scale is None else w.w13_scale.cpu(),
                             None if w.w2_scale is None else w.w2_scale.cpu(), top_k, renorm,
                             rows=rows)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    np.testing.assert_allclose(wts.cpu().numpy(), ref["weights"], rtol=W_RTOL, atol=W_ATOL)
    return assert_out_close(out, ref["out"], rows)


@pytest.mark.parametrize("T,H,I,E,k,renorm,dtype", [
    (4, 128, 256, 8, 2, True, "bf16"),      # tiny bf16 workload
    (4, 128, 256, 8, 2, True, "fp8"),
    (37, 256, 384, 8, 2, True, "fp8"),      # ragged token count
    (200, 512, 256, 16, 4, False, "fp8"),   # several row tiles per expert
    (1, 256, 128, 4, 1, True, "fp8"),
    (9, 128, 128, 1, 1, True, "fp8"),       # single expert: plain SwiGLU MLP
    (9, 128, 128, 1, 1, False, "bf16"),
    (16, 128, 256, 6, 6, False, "fp8"),     # k = E: dense mixture
    (33, 384, 256, 12, 3, True, "bf16"),
    (600, 256, 128, 4, 2, True, "fp8"),     # >256 rows per expert: split tiles
    (130, 1024, 512, 64, 8, True, "fp8"),
    (8, 256, 2176, 4, 2, True, "fp8"),      # I > 2048: down weights in M by default
    (70, 384, 2304, 16, 3, False, "fp8"),   # ragged rows, I > 2048
    (1000, 256, 512, 4, 2, True, "fp8"),    # 500 rows per expert: gate/up on SM pairs
    (3, 256, 256, 1024, 4, True, "bf16"),   # the largest E: routing outside the one-CTA front
    (500, 128, 128, 1024, 8, True, "fp8"),  # the largest E, 4000 pairs over about 980 experts
    (50, 128, 256, 64, 40, False, "fp8"),   # k = 40 of 64
])
@pytest.mark.parametrize("path", ["auto", "weights_in_m", "one_kernel"])
def test_fused_small(gpu_lib, T, H, I, E, k, renorm, dtype, path):
    """The kernel sequence in both placements and, for batches of up to 2048
    pairs, the single cooperative kernel must compute the same layer."""
    w = inputs.make_weights(H, I, E, dtype, seed=T)
    a = inputs.make_activations(T, H, E, "uniform", seed=T)
    flags = {"auto": 0, "weights_in_m": gpu_lib.MOE_FLAG_WEIGHTS_IN_M,
             "one_kernel": gpu_lib.MOE_FLAG_ONE_KERNEL}[path]
    run_case(gpu_lib, w, a, k, renorm, repeat=2, flags=flags)


@pytest.mark.parametrize("T,H,I,E,k", [
    (2600, 256, 128, 16, 2),    # > 4096 pairs: two-pass alignment, tokens quantised once
    (2048, 1024, 128, 32, 8),   # pairs x H > 8M: combine through per-pair rows
    (2048, 1152, 128, 32, 8),   # the same with H % 256 != 0: one weight block per tile
    (512, 4096, 256, 16, 8),    # rows per pair at <= 4096 pairs: one alignment kernel, gather
    (3000, 1024, 256, 8, 4),    # skewed counts: experts with odd numbers of row tiles
    (2500, 1280, 128, 6, 3),    # ragged tiles, five column blocks of 256
])
@pytest.mark.parametrize("placement", ["auto", "weights_in_m"])
def test_fused_large_batch_paths(gpu_lib, T, H, I, E, k, placement):
    w = inputs.make_weights(H, I, E, "fp8", seed=T)
    a = inputs.make_activations(T, H, E, "zipf", seed=T)
    flags = gpu_lib.MOE_FLAG_WEIGHTS_IN_M if placement == "weights_in_m" else 0
    run_case(gpu_lib, w, a, k, True, rows=None, flags=flags)


# Wide gate/up tiles (I % 256 == 0, experts averaging at least 128 rows) run on
# SM pairs (tcgen05 cta_group::2) by default; MOE_FLAG_NO_SM_PAIRS runs the
# gate/up GEMM on one SM per tile (256-row tiles from 256 rows per expert on
# average, else 128-row tiles).
@pytest.mark.parametrize("T,H,I,E,k,routing", [
    (1200, 256, 512, 4, 2, "uniform"),    # one alignment kernel, gather
    (700, 256, 512, 8, 2, "uniform"),     # 175 rows per expert: pairs from 128 on average
    (1100, 384, 768, 4, 3, "uniform"),    # ragged tiles, three weight-block pairs
    (3000, 256, 512, 8, 2, "zipf"),       # > 4096 pairs: two-pass alignment, skew
])
@pytest.mark.parametrize("pairs", [True, False])
def test_fused_wide_tiles_sm_pairs(gpu_lib, T, H, I, E, k, routing, pairs):
    w = inputs.make_weights(H, I, E, "fp8", seed=T)
    a = inputs.make_activations(T, H, E, routing, seed=T)
    run_case(gpu_lib, w, a, k, True, repeat=2,
             flags=0 if pairs else gpu_lib.MOE_FLAG_NO_SM_PAIRS)


# bf16 weights on the large-batch paths: two-pass alignment, bf16 rows of x,
# 256-token gate/up tiles on one SM (SM pairs are FP8 only), combine through the
# fp32 buffer or through rows per pair (P x H > 8M).
@pytest.mark.parametrize("T,H,I,E,k", [(5000, 256, 256, 8, 2), (2048, 1024, 128, 32, 8)])
def test_fused_bf16_large_batch_paths(gpu_lib, T, H, I, E, k):
    w = inputs.make_weights(H, I, E, "bf16", seed=T)
    a = inputs.make_activations(T, H, E, "zipf", seed=T)
    run_case(gpu_lib, w, a, k, True, rows=None)


# More shapes through the SM-pair kernel, drawn once with random.Random(2026):
# E in {2..8}, k <= min(E, 4), H = 128..512, I = 256..1024 (multiples of 256),
# 260..700 routed rows per expert on average, uniform or Zipf routing.
@pytest.mark.parametrize("T,H,I,E,k,routing", [
    (567, 128, 512, 2, 2, "zipf"), (522, 512, 512, 8, 4, "uniform"),
    (265, 128, 1024, 2, 2, "zipf"), (876, 512, 768, 4, 2, "zipf"),
    (3270, 384, 256, 6, 1, "zipf"), (272, 256, 768, 4, 4, "zipf"),
])
def test_fused_sm_pairs_random_shapes(gpu_lib, T, H, I, E, k, routing):
    w = inputs.make_weights(H, I, E, "fp8", seed=T + I)
    a = inputs.make_activations(T, H, E, routing, seed=T + I)
    run_case(gpu_lib, w, a, k, True)


# The unswapped placement (tokens in the MMA M slot, weight rows in N): the
# ablation of the operand swap must compute the same layer.
@pytest.mark.parametrize("T,H,I,E,k,renorm,dtype", [
    (4, 128, 256, 8, 2, True, "bf16"),
    (37, 256, 384, 8, 2, True, "fp8"),
    (200, 512, 256, 16, 4, False, "fp8"),
    (600, 256, 128, 4, 2, True, "fp8"),     # several 128-row tiles per expert
    (130, 1024, 512, 64, 8, True, "fp8"),
    (9, 128, 128, 1, 1, False, "bf16"),
])
def test_fused_tokens_in_m(gpu_lib, T, H, I, E, k, renorm, dtype):
    w = inputs.make_weights(H, I, E, dtype, seed=T)
    a = inputs.make_activations(T, H, E, "uniform", seed=T)
    run_case(gpu_lib, w, a, k, renorm, repeat=2, flags=gpu_lib.MOE_FLAG_TOKENS_IN_M)


@pytest.mark.parametrize("T,H,I,E,k", [(2600, 256, 128, 16, 2), (2048, 1024, 128, 32, 8)])
def test_fused_tokens_in_m_large_batch_paths(gpu_lib, T, H, I, E, k):
    w = inputs.make_weights(H, I, E, "fp8", seed=T)
    a = inputs.make_activations(T, H, E, "zipf", seed=T)
    run_case(gpu_lib, w, a, k, True, rows=None,
             flags=gpu_lib.MOE_FLAG_TOKENS_IN_M)


# Each path switch of the layer, taken on both sides of its threshold (the
# plan is chosen per call from the shape and the routing statistics):
@pytest.mark.parametrize("T,H,I,E,k,dtype", [
    (16, 256, 256, 8, 2, "fp8"),      # at most 16 tokens: one-CTA front
    (17, 256, 256, 8, 2, "fp8"),      # 17: router + alignment kernels
    (8, 256, 256, 256, 4, "fp8"),     # E = 256: one-CTA front
    (8, 256, 256, 257, 4, "fp8"),     # E = 257: router + alignment kernels
    (2048, 256, 256, 8, 2, "fp8"),    # 4096 pairs: one alignment kernel, rows gathered
    (4097, 256, 256, 8, 1, "fp8"),    # 4097 pairs: two-pass alignment, x quantised once per token
    (4096, 2048, 128, 16, 1, "fp8"),  # pairs x H = 8M: fp32 reductions into the combine buffer
    (4096, 2176, 128, 16, 1, "fp8"),  # pairs x H > 8M: bf16 rows per pair, then the row sum
    (254, 128, 512, 4, 2, "fp8"),     # 127 rows per expert on average: single-SM gate/up tiles
    (256, 128, 512, 4, 2, "fp8"),     # 128 rows per expert on average: SM pairs
    (64, 256, 2048, 4, 2, "fp8"),     # I = 2048: down GEMM with tokens in M
    (64, 256, 2176, 4, 2, "fp8"),     # I = 2176: down GEMM with the weights in M
    (17, 256, 256, 8, 2, "bf16"),     # the bf16 path past the one-CTA front
])
def test_fused_path_boundaries(gpu_lib, T, H, I, E, k, dtype):
    w = inputs.make_weights(H, I, E, dtype, seed=T + E)
    a = inputs.make_activations(T, H, E, "uniform", seed=T + E)
    run_case(gpu_lib, w, a, k, True, rows=None)


# Shapes drawn once with random.Random(20261203): E from 1 to 96, k <= min(E, 8),
# H and I multiples of 128 up to 1024 / 1280, T from 1 to 2500, FP8 or bf16,
# uniform or Zipf routing, with and without renormalisation (the oracle's work
# kept under 4 G multiply-adds per case).
RANDOM_SHAPES = [
    (16, 384, 640, 3, 1, False, "fp8", "uniform"), (100, 640, 1152, 8, 3, False, "bf16", "uniform"),
    (100, 1024, 128, 1, 1, True, "fp8", "zipf"), (17, 640, 640, 8, 5, True, "fp8", "zipf"),
    (2500, 384, 256, 2, 2, False, "fp8", "uniform"), (100, 640, 1280, 3, 2, True, "bf16", "uniform"),
    (2, 1024, 896, 96, 1, True, "fp8", "uniform"), (7, 1024, 384, 96, 7, True, "fp8", "zipf"),
    (3, 512, 256, 32, 5, True, "fp8", "uniform"), (7, 640, 512, 13, 4, True, "bf16", "uniform"),
    (17, 768, 512, 1, 1, False, "fp8", "zipf"), (17, 384, 768, 32, 6, True, "fp8", "uniform"),
    (2, 128, 384, 96, 8, False, "fp8", "uniform"), (16, 128, 1152, 1, 1, False, "fp8", "zipf"),
    (1500, 384, 1152, 8, 1, True, "fp8", "uniform"), (2, 384, 128, 96, 1, False, "fp8", "zipf"),
    (17, 384, 1152, 2, 2, True, "fp8", "zipf"), (100, 128, 640, 13, 8, False, "bf16", "uniform"),
    (100, 1024, 512, 2, 2, False, "fp8", "uniform"), (1, 896, 256, 32, 8, False, "fp8", "uniform"),
    (1, 768, 1024, 2, 2, False, "fp8", "zipf"), (17, 768, 896, 96, 2, True, "bf16", "zipf"),
    (7, 896, 256, 96, 2, True, "fp8", "uniform"), (3, 384, 1280, 2, 2, True, "bf16", "uniform"),
]


@pytest.mark.parametrize("T,H,I,E,k,renorm,dtype,routing", RANDOM_SHAPES)
def test_fused_random_shapes(gpu_lib, T, H, I, E, k, renorm, dtype, routing):
    w = inputs.make_weights(H, I, E, dtype, seed=T * 7 + I)
    a = inputs.make_activations(T, H, E, routing, seed=T * 7 + I)
    run_case(gpu_lib, w, a, k, renorm, rows=None)


def test_fused_zipf_skew(gpu_lib):
    T, H, I, E, k = 300, 256, 256, 64, 8
    w = inputs.make_weights(H, I, E, "fp8", seed=5)
    a = inputs.make_activations(T, H, E, "zipf", seed=5)
    run_case(gpu_lib, w, a, k, True)


def test_fused_zero_tokens(gpu_lib):
    w = inputs.make_weights(128, 128, 4, "fp8", seed=1, device="cuda")
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    lg = torch.empty(0, 4, device="cuda")
    out = gpu_lib.moe_fused_forward(x, lg, w.w13, w.w2, w.w13_scale, w.w2_scale, 2, True)
    assert out.shape == (0, 128)


def test_fused_token_permutation(gpu_lib):
    T, H, I, E, k = 50, 256, 256, 8, 2
    w = inputs.make_weights(H, I, E, "fp8", seed=2, device="cuda")
    a = inputs.make_activations(T, H, E, "uniform", seed=2, device="cuda")
    perm = torch.randperm(T, device="cuda")
    o1 = gpu_lib.moe_fused_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
    o2 = gpu_lib.moe_fused_forward(a.x[perm].contiguous(), a.logits[perm].contiguous(), w.w13,
                                   w.w2, w.w13_scale, w.w2_scale, k, True)
    torch.cuda.synchronize()
    d = (o2.float() - o1[perm].float()).abs().max().item()
    assert d <= 2e-2 * o1.float().abs().max().item()


# ---------------------------------------------------------------- full sizes
_WCACHE = {}


def _weights(name):
    if name not in _WCACHE:
        _WCACHE.clear()
        c = inputs.workload(name)
        _WCACHE[name] = inputs.make_weights(c["H"], c["I"], c["E"], c["dtype"], seed=0,
                                            device="cuda")
    return _WCACHE[name]


FULL = [("decode_e8_top2", 1), ("decode_e8_top2", 8), ("decode_e8_top2", 64),
        ("finegrained_e128", 1), ("finegrained_e128", 16), ("finegrained_e128", 256),
        ("skewed_e256", 1), ("skewed_e256", 32), ("skewed_e256", 128),
        ("prefill_e128_uniform", 2048), ("prefill_e128_zipf", 2048)]


@pytest.mark.parametrize("name,T", FULL)
def test_fused_full_size(gpu_lib, name, T):
    """Every output row, element by element, at the measured sizes (stream-K
    splits, split gate/up tiles and per-expert tiles fail locally)."""
    c = inputs.workload(name)
    w = _weights(name)
    a = inputs.make_activations(T, c["H"], c["E"], c["routing"], seed=0, device="cuda")
    run_case(gpu_lib, w, a, c["top_k"], True, rows=None)


@pytest.mark.parametrize("name,T", [("decode_e8_top2", 1), ("decode_e8_top2", 64),
                                    ("finegrained_e128", 256), ("skewed_e256", 128)])
def test_fused_full_size_one_kernel(gpu_lib, name, T):
    """The single cooperative kernel on the small-batch workloads, every row."""
    c = inputs.workload(name)
    w = _weights(name)
    a = inputs.make_activations(T, c["H"], c["E"], c["routing"], seed=0, device="cuda")
    run_case(gpu_lib, w, a, c["top_k"], True, rows=None, flags=gpu_lib.MOE_FLAG_ONE_KERNEL)


@pytest.mark.parametrize("name,T", [("decode_e8_top2", 1), ("decode_e8_top2", 64),
                                    ("finegrained_e128", 16), ("prefill_e128_uniform", 2048)])
def test_fused_full_size_tokens_in_m(gpu_lib, name, T):
    c = inputs.workload(name)
    w = _weights(name)
    a = inputs.make_activations(T, c["H"], c["E"], c["routing"], seed=0, device="cuda")
    run_case(gpu_lib, w, a, c["top_k"], True, rows=None, flags=gpu_lib.MOE_FLAG_TOKENS_IN_M)


def rows_over_every_expert(logits, top_k, E, n, seed):
    """Token rows that cover every expert's segment: the first and the last
    token routed to each expert (routing from the oracle), topped up with
    random tokens to n rows."""
    ids, _ = oracle.route_topk(logits, top_k, True)
    T = ids.shape[0]
    pick = set()
    for e in range(E):
        toks = np.nonzero((ids == e).any(axis=1))[0]
        if len(toks):
            pick.update((int(toks[0]), int(toks[-1])))
    rng = np.random.default_rng(seed)
    rest = [t for t in rng.permutation(T).tolist() if t not in pick]
    pick.update(rest[:max(0, n - len(pick))])
    return sorted(pick)


def test_fused_prefill_8192_rows_over_every_expert(gpu_lib):
    name = "prefill_e128_uniform"
    c = inputs.workload(name)
    w = _weights(name)
    a = inputs.make_activations(8192, c["H"], c["E"], c["routing"], seed=0, device="cuda")
    rows = rows_over_every_expert(a.logits.cpu(), c["top_k"], c["E"], 512, seed=1)
    assert len(rows) >= 512
    run_case(gpu_lib, w, a, c["top_k"], True, rows=rows)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill_e128_uniform", "prefill_e128_zipf"])
def test_fused_prefill_8192(gpu_lib, name):
    c = inputs.workload(name)
    w = _weights(name)
    a = inputs.make_activations(8192, c["H"], c["E"], c["routing"], seed=0, device="cuda")
    run_case(gpu_lib, w, a, c["top_k"], True, rows=None)


# Far past the measured workloads: 65,536 tokens x top-8 = 524,288 pairs (512
# alignment chunks, thousands of row tiles, rows per pair), Zipf routing, outputs
# on 256 rows that cover every expert's segment.  bf16 weights: the oracle forms
# only the sampled rows; FP8 with small H and I: the oracle forms h for every
# pair, since the scale of h spans them all.
@pytest.mark.slow
@pytest.mark.parametrize("T,H,I,E,k,dtype", [
    (65536, 1024, 512, 64, 8, "bf16"),
    (65536, 256, 256, 32, 8, "fp8"),
])
def test_fused_far_past_the_workloads(gpu_lib, T, H, I, E, k, dtype):
    w = inputs.make_weights(H, I, E, dtype, seed=21, device="cuda")
    a = inputs.make_activations(T, H, E, "zipf", seed=21)
    rows = rows_over_every_expert(a.logits, k, E, 256, seed=2)
    run_case(gpu_lib, w, a, k, True, rows=rows)


# (64, 256, 2176, 8, 2): single-SM kernels; (1024, 256, 512, 2, 2): 1024 rows
# per expert, so the gate/up GEMM runs 256-token tiles on SM pairs.
@pytest.mark.parametrize("T,H,I,E,k", [(64, 256, 2176, 8, 2), (1024, 256, 512, 2, 2)])
def test_fused_timed_and_traced_call(gpu_lib, T, H, I, E, k):
    """moe_fused_forward_timed: eight events bracket the steps in order and the
    output agrees with the untimed call's; MOE_DEBUG_TRACE: every CTA of the two
    expert GEMMs that ran leaves stamps with entry and "inputs ready" before
    "first stage landed" and exit."""
    w = inputs.make_weights(H, I, E, "fp8", seed=9, device="cuda")
    a = inputs.make_activations(T, H, E, "uniform", seed=9, device="cuda")
    ws = gpu_lib.alloc_workspace(T, H, I, E, k, gpu_lib.MOE_DT_FP8_E4M3)
    ws.zero_()  # trace rows of CTAs that are not launched stay as they were
    ev = gpu_lib.make_step_events()
    o1 = gpu_lib.moe_fused_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True,
                                   workspace=ws, events=ev, debug_flags=gpu_lib.MOE_DEBUG_TRACE)
    torch.cuda.synchronize()
    assert gpu_lib.moe_check_status(ws) == 0
    times = [ev[0].elapsed_time(e) for e in ev]
    assert all(t1 >= t0 for t0, t1 in zip(times, times[1:]))
    tr = gpu_lib.read_trace(ws, T, H, I, E, k, gpu_lib.MOE_DT_FP8_E4M3).numpy()
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    for g in range(2):
        rows = tr[g][:n_sm]  # at most one CTA per SM
        stamps = rows[np.all(rows > 0, axis=1)]  # CTAs that ran at least one stage
        assert len(stamps) > 0
        entry, ready, first, leave = (stamps[:, i] for i in range(4))
        assert np.all(entry <= ready) and np.all(ready <= leave)
        assert np.all(entry <= first) and np.all(first <= leave)
    o2 = gpu_lib.moe_fused_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True,
                                   workspace=ws)
    torch.cuda.synchronize()
    d = (o1.float() - o2.float()).abs().max().item()
    assert d <= 2e-2 * o2.float().abs().max().item()
