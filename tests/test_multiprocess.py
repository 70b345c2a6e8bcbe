"""The N > 1 host path of bench.py on CPU, world size 2 over gloo: the path
has no data exchange (independent replicas, weak scaling), so what runs on
several GPUs is the barrier around the timed region, the max of the timed
milliseconds over ranks, the per-rank input seeds and the rule that only
rank 0 prints (the other ranks of the reference arm exit without work)."""
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_setup(world)
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(ws)
        # each rank timed a different duration: everyone must see the slowest
        t = bench.max_over_ranks(ws, 10.0 + 5.0 * rank, torch.device("cpu"))
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_two_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_replicas_draw_different_inputs():
    from exact_tiled_attention_10_gb300.inputs import qkv
    a = qkv(1, 2, 64, 64, 1003 + 0)[0]
    b = qkv(1, 2, 64, 64, 1003 + 1000)[0]  # rank 1's seed offset in bench.Step
    assert not torch.equal(a, b)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    assert buf.getvalue() == ""
