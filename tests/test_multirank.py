"""The multi-rank host logic of bench.py on CPU with the gloo backend,
world size 2 (the GPU path runs one replica per rank with no data-path
collective; only the timing reduction crosses ranks)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

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
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        mine = [10.0, 12.5][rank]  # rank 1 is the slower one
        slowest = bench.max_over_ranks(mine, dist, "cpu")
        value = bench.job_value(world, 268_451_904 * 32, 100, slowest * 100)
        # the reference arm prints on rank 0 only; other ranks return at once
        buf = io.StringIO()
        if rank == 1:
            with redirect_stdout(buf):
                bench.reference_arm(None, rank, world)
        q.put((rank, slowest, value, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_and_count_both():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, value, out in got:
        assert slowest == 12.5
        # both ranks' bytes over the slower rank's time (12.5 ms per step)
        assert value == pytest.approx(2 * 268_451_904 * 32 / 12.5e-3 / 1e9)
        assert out == ""
