"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
gets its own batch (distinct seeds, same weights), the reported time is the
slowest rank's, and the whole-job value sums the ranks' work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from nvfp4_quantized_linear_gb300 import synthetic as syn
    local_time = 0.010 * (rank + 1)                    # rank 1 is the slow one
    slowest = bench.max_over_ranks(local_time, "cpu")
    probs = bench.layer_problems(bench.DEFAULT_WORKLOAD, 16, rank)
    x = syn.make_activation(probs[0])
    w = syn.bf16_normal((probs[0].n, probs[0].k), 0.02, probs[0].seed + 100_000)
    seeds = [p.seed for p in probs]
    gathered = [None] * world
    dist.all_gather_object(gathered, (seeds, float(x.float().sum()), float(w.float()[:4, :4].sum())))
    value = bench.aggregate(sum(p.flops for p in probs), world, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, gathered, value))


def test_two_gloo_ranks_shard_batches_and_take_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    (_, slow0, g0, v0), (_, slow1, g1, v1) = res
    assert slow0 == slow1 == pytest.approx(0.020)
    assert g0 == g1
    (seeds_a, xa, _), (seeds_b, xb, _) = g0
    assert set(seeds_a).isdisjoint(seeds_b)        # distinct per-rank batches
    assert xa != xb
    import bench
    flops = sum(p.flops for p in bench.layer_problems(bench.DEFAULT_WORKLOAD, 16, 0))
    assert v0 == v1 == pytest.approx(flops * 2 / 0.020)


def test_rank_seed_and_aggregate_single_process():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_seed(1000, 0) == 1000 and bench.rank_seed(1000, 1) != 1000
    assert bench.aggregate(10.0, 4, 2.0) == 20.0
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.quant_bytes(16, 256) == 2 * 16 * 256 + 16 * 128 + 128 * 16
