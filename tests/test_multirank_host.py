"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks.  The path shards over sequences as
independent replicas (no collective on the data path); only the timing bookkeeping crosses ranks:
a barrier, the max of the ranks' times, and the whole-job throughput over all replicas' bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads as W
        # each replica draws its own inputs of the same shapes
        lens = [20, 33, 47]
        inp = W.device_decode_inputs(lens, n_q_heads=8, n_kv_heads=2, head_dim=64, block_size=16,
                                     dtype=torch.float32, num_blocks=16, max_blocks_per_seq=4, device="cpu",
                                     seed=bench.replica_seed(rank), layers=1)
        bench.barrier(dist, cuda=False)
        my_ms = 10.0 + 5.0 * rank  # a replica's timed region
        slowest = bench.max_over_ranks(my_ms, dist, device="cpu")
        value = bench.whole_job_gbs(1e9, 100, world, slowest)
        qs = [torch.zeros_like(inp["q"]) for _ in range(world)]
        dist.all_gather(qs, inp["q"])
        out.put((rank, slowest, value, [tuple(q.shape) for q in qs], bool(torch.equal(qs[0], qs[1]))))
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_time_and_the_whole_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, shapes, same in results:
        assert slowest == 15.0                      # max over ranks
        assert value == pytest.approx(1e9 * 100 * 2 / 15e-3 / 1e9)  # all replicas' bytes / slowest time
        assert shapes[0] == shapes[1]               # same shapes on every replica
        assert not same                             # different values on every replica


def test_single_process_path_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.whole_job_gbs(2e9, 10, 1, 1000.0) == pytest.approx(20.0)
