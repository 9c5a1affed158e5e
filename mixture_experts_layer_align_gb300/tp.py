"""Tensor-parallel sharding of the fused MoE layer over the intermediate size.

The pages measure their TTFT gain at 8-way tensor parallelism ("Triton JIT
recompilation elimination", English original page); the layer shards over
the expert MLP's intermediate size I:

  rank r of W holds, for every expert, the gate rows [r I/W, (r+1) I/W) and
  the up rows [I + r I/W, I + (r+1) I/W) of w13, and the columns
  [r I/W, (r+1) I/W) of w2 (per-expert weight scales are unchanged: the codes
  are the same bytes);
  routing is replicated: every rank sees the same x and router logits;
  every rank runs the unchanged single-GPU layer on its shard, whose output
  is the partial sum over its slice of I of the down projection (SiLU*up is
  elementwise in I, so the slices are independent);
  one all-reduce (sum) of the [T, H] output follows.

The per-tensor FP8 scale of h spans the whole h: each rank runs the layer
as two calls of the library and max-reduces the one fp32 max |h| word of its
workspace between them, so every rank quantises its slice of h exactly as
the unsharded layer would (with each rank's own scale the summed result
drifts outside the FP8 tolerance, see the CPU oracle's sharded test).
Requires (I / W) % 128 == 0 (the kernels' K tile).  This module only slices
tensors and calls the library and torch.distributed; all arithmetic of the
layer runs in the CUDA kernels.
"""
from __future__ import annotations


def shard_weights(w13, w2, rank: int, world: int):
    """(w13 [E, 2 I/W, H], w2 [E, H, I/W]) of rank `rank`, contiguous copies."""
    import torch
    E, two_i, H = w13.shape
    I = two_i // 2
    if world < 1 or not 0 <= rank < world or I % world != 0:
        raise ValueError(f"I={I} does not split over {world} ranks")
    n = I // world
    lo, hi = rank * n, (rank + 1) * n
    w13_r = torch.cat([w13[:, lo:hi, :], w13[:, I + lo:I + hi, :]], dim=1).contiguous()
    w2_r = w2[:, :, lo:hi].contiguous()
    return w13_r, w2_r


def tp_forward(x, router_logits, w13_r, w2_r, w13_scale, w2_scale, top_k: int,
               renormalize: bool = True, group=None, workspace=None, stream=None):
    """This rank's shard of the layer: the gate/up call, an all-reduce (max)
    of the max |h| word, the down call, then the all-reduce (sum) of the
    output rows over `group` (fp32 sum of the ranks' bf16 partial outputs).
    Without an initialised process group it runs the shard alone.  Returns
    bf16 [T, H]."""
    import torch
    import torch.distributed as dist
    from . import (MOE_DT_BF16, MOE_DT_FP8_E4M3, alloc_workspace, h_amax_view,
                   moe_fused_forward_down, moe_fused_forward_gate_up)
    T, H = x.shape
    E = router_logits.shape[1]
    I = w13_r.shape[1] // 2
    if workspace is None:
        workspace = alloc_workspace(T, H, I, E, top_k,
                                    MOE_DT_FP8_E4M3 if w13_scale is not None else MOE_DT_BF16,
                                    x.device)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    parallel = dist.is_available() and dist.is_initialized()
    moe_fused_forward_gate_up(x, router_logits, w13_r, w2_r, w13_scale, w2_scale, top_k,
                              renormalize, out, workspace, stream)
    if parallel and w13_scale is not None:
        dist.all_reduce(h_amax_view(workspace), op=dist.ReduceOp.MAX, group=group)
    moe_fused_forward_down(x, router_logits, w13_r, w2_r, w13_scale, w2_scale, top_k,
                           renormalize, out, workspace, stream)
    acc = out.float()
    if parallel:
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    return acc.to(torch.bfloat16)


__all__ = ["shard_weights", "tp_forward"]
