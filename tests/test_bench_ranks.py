"""The multi-process bookkeeping of bench.py (one process per GPU, no data
exchange): barriers, maximum over ranks, a schedule pick that every rank
agrees on, and whole-job rates, checked with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r = bench.Ranks(dist, "cpu")
        r.barrier()
        # per-rank times: rank 1 is the slow one
        mx = r.max(2.0 + 3.0 * rank)
        # each rank alone would pick differently; the max over ranks decides
        trials = {"shift": 1.0 if rank == 0 else 9.0, "symmetric_shift": 5.0, "descending_q": 7.0 - rank}
        pick = r.pick_fastest(trials)
        tie = r.pick_fastest({"a": 4.0, "b": 4.0})
        rate = r.rate(10.0, mx)
        out.put((rank, r.world, r.rank, mx, pick, tie, rate))
        r.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, rr, mx, pick, tie, rate) in enumerate(res):
        assert (r, w, rr) == (rank, world, rank)
        assert mx == 5.0                       # the slowest rank's time
        assert pick == "symmetric_shift"      # worst case 5 beats max(1, 9) and max(7, 6)
        assert tie == "a"                      # ties go to the first key, on every rank
        assert rate == pytest.approx(world * 10.0 / 5e-3)   # work of all ranks over the slowest time


def test_one_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks()
    r.barrier()
    assert (r.world, r.rank) == (1, 0)
    assert r.max(3) == 3.0
    assert r.pick_fastest({"x": 2.0, "y": 1.0}) == "y"
    assert r.rate(4.0, 2.0) == pytest.approx(2000.0)


def test_pick_fastest_keeps_the_preferred_schedule_within_the_margin():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks()
    trials = {"symmetric_shift": 8.6867, "shift": 8.6792, "descending_q": 14.3}
    assert r.pick_fastest(trials) == "shift"
    assert r.pick_fastest(trials, prefer="symmetric_shift") == "symmetric_shift"
    assert r.pick_fastest({"a": 10.0, "b": 9.0}, prefer="a") == "b"   # 11% slower: not kept
    assert r.pick_fastest({"a": 10.0, "b": 9.0}, prefer="zzz") == "b"
