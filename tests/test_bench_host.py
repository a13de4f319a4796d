"""Host-side logic of bench.py that needs no GPU: argument defaults, and the replica
aggregation (max time, summed units) over a world-size-2 gloo group on CPU."""
import os
import socket

import torch.multiprocessing as mp

import bench


def test_defaults():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    t, u = bench.aggregate(elapsed_s=1.0 + rank, units=10.0 * (rank + 1), dist=dist)
    bench.barrier(dist)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_replica_aggregation_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the max time (2.0 s) and the total units (10 + 20)
    assert out == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_single_process_aggregation_is_identity():
    assert bench.aggregate(1.5, 7.0, None) == (1.5, 7.0)
