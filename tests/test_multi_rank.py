"""The bench's N > 1 path on the CPU: two gloo ranks exercise the barrier, the
max-over-ranks reduction of the timings, the whole-job (weak-scaling) rate
and the rank-0-only output, as `torchrun --nproc-per-node 2 bench.py` uses
them on GPUs."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        w, r, local = bench.dist_env()
        bench.rank_barrier(w)
        times = bench.max_over_ranks([10.0 + rank, 5.0 - rank, 1.0 * rank], w)
        rate = bench.job_rate(w, 1_000_000, 100, times[0])
        q.put((r, local, w, times, rate, bench.prints(r)))
        bench.rank_barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, local, w, times, rate, printing) in enumerate(res):
        assert (r, local, w) == (rank, rank, ws)
        # every rank sees the maximum over ranks of each timing
        assert times == [11.0, 5.0, 1.0]
        # whole-job rate: both ranks' bytes over the slowest rank's time
        assert rate == pytest.approx(2 * 1_000_000 * 100 / 11e-3 / 1e9)
        assert printing == (rank == 0)


def test_single_rank_helpers_need_no_process_group():
    assert bench.max_over_ranks([3.0, 1.0], 1) == [3.0, 1.0]
    bench.rank_barrier(1)
    assert bench.job_rate(1, 2e9, 10, 1000.0) == pytest.approx(20.0)
    assert bench.prints(0) and not bench.prints(1)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"workload": "fixed_tree", "steps": 1, "warmup": 0})()
    bench.run_reference(args)          # returns at once: rank 1 neither computes nor prints
    assert capsys.readouterr().out == ""
