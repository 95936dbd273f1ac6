"""The multi-rank benchmark path, on CPU with the gloo backend (world size 2):
each rank runs an independent replica (its own seed), and the whole-job
figures are the slowest rank's time and the sum of all ranks' bytes."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w = bench.workload("tiny_decode", rank, None)
    maxes, sums = bench.reduce_over_ranks([1.0 + rank, 10.0 * (rank + 1)], [w.kv_bytes(), w.total_q],
                                          world, torch.device("cpu"))
    out.put((rank, maxes, sums, w.key_cache.view(np.uint16)[:2, 0, 0, :4].tolist()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_reduce_max_time_and_sum_bytes():
    import bench
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w0 = bench.workload("tiny_decode", 0, None)
    for rank, maxes, sums, _ in res:
        assert maxes == [2.0, 20.0]                      # slowest rank
        assert sums == [2.0 * w0.kv_bytes(), 2.0 * w0.total_q]  # both replicas
    # the replicas are different draws (seed = rank), not copies
    assert res[0][3] != res[1][3]


def test_single_rank_passes_through():
    import bench
    assert bench.reduce_over_ranks([1.5], [7], 1, None) == ([1.5], [7])
