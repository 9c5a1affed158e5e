"""Tensor-parallel sharding of the layer over the intermediate size I (the
8-way tensor-parallel setting of "Triton JIT recompilation elimination",
English original page), checked on the CPU with two gloo ranks.

Each rank holds the gate and up rows and the w2 columns of its slice of I
(sliced here with numpy, independently of the package's shard_weights);
routing is replicated.  Rank r runs the oracle on its shard; the max |h| of
the ranks is max-reduced so that every rank quantises h with the scale of
the whole tensor; the ranks' partial outputs are sum-reduced.  The sum must
equal the unsharded oracle to fp64 rounding (the slices of I are
independent until the down projection, whose sum over I is split by rank).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from mixture_experts_layer_align_gb300 import inputs

CASES = [("fp8", 9, 256, 512, 8, 2), ("bf16", 5, 128, 256, 4, 2)]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _numpy_shard(w13, w2, rank, world):
    w13 = np.asarray(w13)
    w2 = np.asarray(w2)
    I = w13.shape[1] // 2
    n = I // world
    lo, hi = rank * n, (rank + 1) * n
    return (np.ascontiguousarray(np.concatenate([w13[:, lo:hi], w13[:, I + lo:I + hi]], axis=1)),
            np.ascontiguousarray(w2[:, :, lo:hi]))


def _bits(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for dtype, T, H, I, E, k in CASES:
            w = inputs.make_weights(H, I, E, dtype, seed=7)
            a = inputs.make_activations(T, H, E, "uniform", seed=7)
            w13_r, w2_r = _numpy_shard(_bits(w.w13), _bits(w.w2), rank, world)
            if dtype == "bf16":
                w13_r = torch.from_numpy(w13_r.view(np.int16)).view(torch.bfloat16)
                w2_r = torch.from_numpy(w2_r.view(np.int16)).view(torch.bfloat16)
            # pass 1: this shard's max |h|, max-reduced over the ranks
            local = oracle.moe_forward(a.x, a.logits, w13_r, w2_r, w.w13_scale, w.w2_scale, k,
                                       True)
            amax = torch.tensor([local["h_amax"]], dtype=torch.float32)
            dist.all_reduce(amax, op=dist.ReduceOp.MAX)
            # pass 2: the partial output with the scale of the whole tensor
            part = oracle.moe_forward(a.x, a.logits, w13_r, w2_r, w.w13_scale, w.w2_scale, k,
                                      True, h_amax=float(amax.item()) if dtype == "fp8" else None)
            out = torch.from_numpy(part["out"].copy())
            dist.all_reduce(out, op=dist.ReduceOp.SUM)
            per_rank = torch.from_numpy(local["out"].copy())
            dist.all_reduce(per_rank, op=dist.ReduceOp.SUM)
            if rank == 0:
                results[dtype] = (out.numpy(), per_rank.numpy(), float(amax.item()))
    finally:
        dist.destroy_process_group()


def test_sharded_oracle_sums_to_the_unsharded_layer():
    world = 2
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                       join=True, start_method="spawn")
    for dtype, T, H, I, E, k in CASES:
        w = inputs.make_weights(H, I, E, dtype, seed=7)
        a = inputs.make_activations(T, H, E, "uniform", seed=7)
        ref = oracle.moe_forward(a.x, a.logits, w.w13, w.w2, w.w13_scale, w.w2_scale, k, True)
        summed, per_rank_scales, amax = results[dtype]
        scale = np.abs(ref["out"]).max()
        assert np.abs(summed - ref["out"]).max() <= 1e-12 * scale, dtype
        if dtype == "fp8":
            # the max-reduced max |h| is the unsharded one
            assert amax == ref["h_amax"]
            # with each rank's own scale of h the ranks quantise h differently
            # from the unsharded layer (here by 2.9e-2 of max |out|, beyond
            # the FP8 tolerance): the max-reduction is needed
            err = np.abs(per_rank_scales - ref["out"]).max() / scale
            assert err > 1e-3


def test_package_shard_weights_matches_the_slicing():
    """The package's shard_weights (used by tp_forward on the GPU) slices the
    same rows and columns."""
    from mixture_experts_layer_align_gb300 import tp
    w = inputs.make_weights(128, 512, 4, "fp8", seed=3)
    for world in (2, 4):
        for rank in range(world):
            w13_r, w2_r = tp.shard_weights(w.w13, w.w2, rank, world)
            n13, n2 = _numpy_shard(w.w13.numpy(), w.w2.numpy(), rank, world)
            assert np.array_equal(w13_r.numpy(), n13) and np.array_equal(w2_r.numpy(), n2)
            assert w13_r.is_contiguous() and w2_r.is_contiguous()
    with pytest.raises(ValueError):
        tp.shard_weights(w.w13, w.w2, 0, 3)
