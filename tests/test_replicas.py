"""The multi-GPU path of the benchmark is N independent replicas (the layer
has no exchange step): each rank times its own steps, the job time is the
slowest rank's, and the whole-job throughput counts every rank's tokens.
Checked here with two gloo ranks on the CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")  # rank 1 is slower
    q.put((rank, ms, bench.job_tokens_per_s(world, 127, 100, ms), bench.dist_env()))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tps, env in out:
        assert ms == 15.0                          # max over ranks
        assert tps == 2 * 127 * 100 / 15e-3        # both replicas' tokens over the job time
        assert env == (rank, rank, world)


def test_single_process_is_the_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tokens_per_s(1, 10, 4, 2.0) == 20000.0
