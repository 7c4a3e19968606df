"""The N > 1 host path of bench.py on the CPU: two gloo ranks. Each rank times its own
replica of the batch (no data-path collective); the job's time is the maximum over the
ranks and its value the bytes of every rank over that time."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d, r, local, w = bench._dist()
    try:
        res = {"ms_graph": 1.0 + rank, "dec_ms": 0.5 * (world - rank)}
        bench.reduce_max(res, ("ms_graph", "dec_ms"), d, "cpu")
        d.barrier()
        q.put((r, w, res["ms_graph"], res["dec_ms"], bench.job_value(1e9, w, res["ms_graph"])))
    finally:
        d.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
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
    for r, (rank, w, ms, dec, val) in enumerate(out):
        assert (rank, w) == (r, world)
        assert ms == 2.0 and dec == 1.0          # the maxima over the ranks
        assert val == pytest.approx(2 * 1e9 / 2e-3 / 1e9)
