"""The multi-process side of bench.py, on CPU with gloo: with N replicas the
timing is the maximum over ranks and every rank reaches the barrier; the
reference arm runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(0.5 + rank, world)
        w, r, _ = bench.dist_env()
        out[rank] = (t, w, r)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == (1.5, 2, 0)
    assert res[1] == (1.5, 2, 1)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_reference_arm_is_silent_off_rank_0(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert rc == 0 and buf.getvalue() == ""


def test_warmup_below_three_is_refused():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
