"""The N > 1 path of bench.py on CPU: independent replicas whose timings are
reduced with a max over ranks (gloo, world size 2), the whole-job value, and
the reference arm's silence on ranks other than 0."""
import argparse
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # per-rank step times: rank 1 is the slow one in the first entry,
        # rank 0 in the second
        mine = [40.0 + 10.0 * rank, 55.0 - 5.0 * rank]
        got = bench.max_over_ranks(mine, dist, "cpu")
        value = bench.whole_job_value(7.424e13, got[0], world)
        out[rank] = (got, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    for rank in range(world):
        got, value = out[rank]
        assert got == [50.0, 55.0]            # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 7.424e13 / 0.050 / 1e12)  # both ranks' work


def test_single_rank_reduction_is_the_identity():
    assert bench.max_over_ranks([3.0, 4.5], None, "cpu") == [3.0, 4.5]
    assert bench.whole_job_value(1e12, 1000.0, 1) == pytest.approx(1.0)


def test_reference_arm_is_silent_off_rank_0(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(config="tiny", steps=1, warmup=0, ref_heads=1, ref_rows=4)
    assert bench.bench_reference(args) is None
    assert capsys.readouterr().out == ""
