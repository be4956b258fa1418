"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each with its own
batch (weak scaling), the step time is the maximum over ranks and the value
counts the points of every rank.  No GPU and no data-path collective."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    r, lr, ws = bench.dist_env()
    t = 1.0 + rank                      # rank 1 is the slow one
    tmax = bench.max_over_ranks(t, dist)
    seed = bench.rank_seed(1235, r)
    q.put((r, ws, tmax, seed, bench.aggregate(100, ws, tmax)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, t0, s0, v0), (r1, ws1, t1, s1, v1) = res
    assert (r0, r1) == (0, 1) and ws0 == ws1 == 2
    assert t0 == t1 == 2.0                # the slowest rank sets the time
    assert s0 != s1                       # independent batches per rank
    assert v0 == v1 == pytest.approx(100 * 2 / 2.0)


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.max_over_ranks(3.5) == 3.5


def test_algorithmic_bytes_of_the_encoder_step():
    import workloads
    ab = bench.algorithmic_bytes(workloads.WORKLOADS["encoder_train"])
    # value 45.5 MB, locations 45.5 MB, weights 22.8 MB, output 45.5 MB
    assert ab["fwd"] == pytest.approx(159.3e6, rel=2e-3)
    assert ab["bwd"] == pytest.approx(273.1e6, rel=2e-3)
