"""The multi-rank (replica) path of bench.py on CPU: two gloo ranks, as the
driver launches bench.py under torchrun for N > 1.  The data path has no
collective (each rank syncs and runs its own replica); what crosses ranks is
the timing: the maximum over ranks of the timed region and of the weight-sync
phase, and the whole-job value = bytes of all ranks / that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        total, sync, value = bench.aggregate_over_ranks(dist, torch, 10.0 + rank, 1.0 + 0.5 * rank, 2.0e9,
                                                        world, "cpu")
        out.put((rank, total, sync, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_time_and_sum_the_bytes():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, sync, value in res:
        assert total == 11.0 and sync == 1.5           # the slower rank decides
        assert value == pytest.approx(2 * 2.0e9 / 1.5 / 1e6)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    total, sync, value = bench.aggregate_over_ranks(None, torch, 5.0, 2.0, 1.0e9, 1, "cpu")
    assert (total, sync) == (5.0, 2.0) and value == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main_reference(None)  # rank 1 returns before reading any argument
    assert capsys.readouterr().out == ""
