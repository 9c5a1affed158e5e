"""Seeded synthetic inputs for the fused MoE layer.

This module is shared by the GPU path's tests and benchmark and by the CPU
oracle's tests.  It draws random numbers and lays them out; it holds none of
the layer's arithmetic (routing, alignment, GEMMs, activation scaling,
combine).  Weights are produced the way a model loader would hand them to the
layer: fp32 N(0, 0.02) draws, and for FP8 workloads one scale per expert per
weight tensor (amax / 448) with the E4M3 codes produced by torch's own
float8_e4m3fn cast.

Workloads (the sizes of the five measured configurations):
  tiny_bf16           T=4,                 H=128,  I=256,   E=8,   k=2, bf16 weights
  decode_e8_top2      T in 1..64 (x2),     H=4096, I=14336, E=8,   k=2, FP8
  finegrained_e128    T in {1,4,16,64,256}, H=2048, I=768,  E=128, k=8, FP8
  skewed_e256         T in {1,8,32,128},   H=7168, I=2048,  E=256, k=8, FP8, Zipf logits
  prefill_e128        T in {2048,8192},    H=2048, I=768,   E=128, k=8, FP8, uniform or Zipf
All renormalise the top-k weights.  Draw order per case: logits, x (one
generator seeded with (seed, T)), then w13, w2 (a generator seeded with seed
alone, so that one set of weights serves every T of a sweep).

The inverse-rotary / per-head FP8 kernel takes head vectors x ~ N(0,1) bf16
[T, NH, D], positions uniform in [0, max_pos) and the rotary cache a model
would hold: cos and sin of pos * base^(-2i/D), computed in fp64 and stored as
fp32 [max_pos, D/2] (base 10000).
"""
from __future__ import annotations

import dataclasses

import torch

WORKLOADS = {
    "tiny_bf16": dict(H=128, I=256, E=8, top_k=2, dtype="bf16", routing="uniform", T=(4,)),
    "decode_e8_top2": dict(H=4096, I=14336, E=8, top_k=2, dtype="fp8", routing="uniform",
                           T=(1, 2, 4, 8, 16, 32, 64)),
    "finegrained_e128": dict(H=2048, I=768, E=128, top_k=8, dtype="fp8", routing="uniform",
                             T=(1, 4, 16, 64, 256)),
    "skewed_e256": dict(H=7168, I=2048, E=256, top_k=8, dtype="fp8", routing="zipf",
                        T=(1, 8, 32, 128)),
    "prefill_e128_uniform": dict(H=2048, I=768, E=128, top_k=8, dtype="fp8", routing="uniform",
                                 T=(2048, 8192)),
    "prefill_e128_zipf": dict(H=2048, I=768, E=128, top_k=8, dtype="fp8", routing="zipf",
                              T=(2048, 8192)),
}

E4M3_MAX = 448.0
ZIPF_S = 1.1


@dataclasses.dataclass
class Weights:
    """Expert weights as the layer consumes them.

    w13: [E, 2I, H] (rows [0,I) gate, [I,2I) up), w2: [E, H, I].
    FP8: uint8 E4M3 codes plus fp32 per-expert scales.  bf16: bf16 tensors,
    scales None.
    """
    w13: torch.Tensor
    w2: torch.Tensor
    w13_scale: torch.Tensor | None
    w2_scale: torch.Tensor | None
    dtype: str
    H: int
    I: int
    E: int


@dataclasses.dataclass
class Activations:
    x: torch.Tensor        # bf16 [T, H]
    logits: torch.Tensor   # fp32 [T, E]
    T: int


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def zipf_bias(E: int, s: float = ZIPF_S) -> torch.Tensor:
    """2*log(p_e), p_e = (e+1)^-s / sum: expert e's popularity is its rank."""
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    p = ranks.pow(-s)
    p = p / p.sum()
    return (2.0 * torch.log(p)).to(torch.float32)


def make_weights(H: int, I: int, E: int, dtype: str = "fp8", seed: int = 0,
                 device="cpu", std: float = 0.02) -> Weights:
    """Draw w13 then w2 ~ N(0, std) in fp32, expert by expert, and hand them
    over as bf16 or as E4M3 codes with a per-expert scale."""
    g = _gen(device, seed * 1000003 + 17)
    if dtype == "bf16":
        w13 = torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device=device)
        w2 = torch.empty(E, H, I, dtype=torch.bfloat16, device=device)
        for e in range(E):
            w13[e] = (torch.randn(2 * I, H, generator=g, device=device) * std).to(torch.bfloat16)
        for e in range(E):
            w2[e] = (torch.randn(H, I, generator=g, device=device) * std).to(torch.bfloat16)
        return Weights(w13, w2, None, None, "bf16", H, I, E)
    if dtype != "fp8":
        raise ValueError(dtype)
    w13 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
    w2 = torch.empty(E, H, I, dtype=torch.uint8, device=device)
    s13 = torch.empty(E, dtype=torch.float32)
    s2 = torch.empty(E, dtype=torch.float32)
    for dst, scales, shape in ((w13, s13, (2 * I, H)), (w2, s2, (H, I))):
        for e in range(E):
            w = torch.randn(*shape, generator=g, device=device) * std
            s = (w.abs().amax() / E4M3_MAX).to(torch.float32)
            scales[e] = s.item()
            dst[e] = (w / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return Weights(w13, w2, s13.to(device), s2.to(device), "fp8", H, I, E)


def make_activations(T: int, H: int, E: int, routing: str = "uniform", seed: int = 0,
                     device="cpu") -> Activations:
    """logits ~ N(0,1) fp32 (+ Zipf popularity bias), then x ~ N(0,1) as bf16."""
    g = _gen(device, seed * 7919 + T)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if routing == "zipf":
        logits = logits + zipf_bias(E).to(device)
    elif routing != "uniform":
        raise ValueError(routing)
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return Activations(x, logits.contiguous(), T)


@dataclasses.dataclass
class RopeInputs:
    x: torch.Tensor          # bf16 [T, NH, D]
    positions: torch.Tensor  # int32 [T]
    cos: torch.Tensor        # fp32 [max_pos, D/2]
    sin: torch.Tensor        # fp32 [max_pos, D/2]


def make_rope_inputs(T: int, NH: int, D: int, max_pos: int = 8192, seed: int = 0,
                     device="cpu", base: float = 10000.0) -> RopeInputs:
    g = torch.Generator(device="cpu").manual_seed(seed * 7919 + T)
    x = torch.randn(T, NH, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    positions = torch.randint(0, max_pos, (T,), generator=g, dtype=torch.int64).to(torch.int32)
    inv_freq = base ** (-torch.arange(0, D // 2, dtype=torch.float64) * 2.0 / D)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv_freq[None, :]
    return RopeInputs(x.to(device), positions.to(device), torch.cos(ang).float().to(device),
                      torch.sin(ang).float().to(device))


def workload(name: str) -> dict:
    return dict(WORKLOADS[name])


def weight_bytes_per_expert(H: int, I: int, dtype: str) -> int:
    esize = 1 if dtype == "fp8" else 2
    return 3 * H * I * esize


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["WORKLOADS", "Weights", "Activations", "make_weights", "make_activations",
           "zipf_bias", "workload", "weight_bytes_per_expert", "ceil_div", "RopeInputs",
           "make_rope_inputs"]
