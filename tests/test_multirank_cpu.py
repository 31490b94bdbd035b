"""The multi-GPU bench path runs independent replicas: ranks share nothing but a barrier
and the max-over-ranks timing. Exercised here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup(0)          # 0 GPUs: gloo
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
    ms_max = bench.allreduce_max(ms, w)
    q.put((rank, ms_max, bench.aggregate_tokens_per_s(w, 1024, 4, ms_max)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]
    # two replicas, 1024 tokens per step, 4 steps, 15 ms: 2*4096 tokens / 0.015 s
    assert res[0][2] == pytest.approx(2 * 1024 * 4 / 0.015)
