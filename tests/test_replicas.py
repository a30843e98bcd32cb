"""N > 1 is independent replicas: the path shards by problem with no exchange
step, so bench.py under torchrun runs one replica per rank (its own seeded
problem), times each, takes the maximum over ranks and reports the aggregate.
These CPU tests run that host logic as two gloo ranks."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import bench
from nvfp4_quantization_grouped_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    r, w, _ = bench.dist_setup(world)
    slowest = bench.max_over_ranks(10.0 * (r + 1), w)       # each rank's "elapsed ms"
    bench.barrier(w)
    pr = inputs.make_problem("tiny_srelu_mxfp8", r)          # the replica's own seeded problem
    q.put((r, w, slowest, pr.x[:8].tolist(), pr.probs[:8].tolist()))
    dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[2] == 20.0 for g in got)                   # max over ranks, seen by every rank
    assert got[0][3] != got[1][3] and got[0][4] != got[1][4]   # independent problems per rank


def test_aggregate_is_weak_scaling_sum():
    # 2 replicas of 1 GB per step, 10 steps, slowest rank 100 ms: 200 GB/s for the job
    assert np.isclose(bench.aggregate_gbs(2, 1e9, 10, 100.0), 200.0)
    assert np.isclose(bench.aggregate_gbs(1, 1e9, 10, 100.0), 100.0)
