"""The multi-replica path of the benchmark on CPU with two gloo ranks.

The sub-block does not shard (one request per GPU, replicas only): ranks
share nothing but a barrier and the max-over-ranks of their timings, and the
reference arm runs on rank 0 alone.
"""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 7.0 * rank                       # rank 1 is the slow replica
        worst = bench.max_over_ranks(ms, world, "cpu")
        rate = bench.job_throughput(100.0, world, worst)
        dist.barrier()
        # the reference arm: every rank but 0 leaves without work
        import argparse
        from h3inputs import CONFIGS
        args = argparse.Namespace(steps=1, warmup=3, gpus=world)
        rc = bench.run_reference(args, CONFIGS["tiny"]) if rank != 0 else 0
        out.put((rank, worst, rate, rc))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [17.0, 17.0]
    # two replicas x 100 units in 17 ms
    assert all(abs(r[2] - 2 * 100.0 / 17e-3) < 1e-6 for r in res)
    assert res[1][3] == 0
