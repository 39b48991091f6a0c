"""The rule that splits grouped-query tasks per query head (dash_head_split),
checked on the CPU against worker loads computed from the oracle simulator's
own task lists (oracle/dagsim.py builds them independently of the library)."""
import pytest

from oracle import dagsim as G
from tile_scheduling_persistent_gb300 import dash

P = 152


def busiest(schedule, B, Hq, Hkv, n, causal):
    tasks = G.make_tasks(schedule, B, Hq, Hkv, n, causal)
    load = [0] * P
    for k, t in enumerate(tasks):
        load[k % P] += len(t)
    return max(load)


@pytest.mark.parametrize("schedule,causal,B,Hq,Hkv,S,D", [
    ("symmetric_shift", True, 1, 32, 8, 16384, 128),   # the LLaMA3-8B-shaped workload: split
    ("shift", True, 1, 32, 8, 16384, 128),
    ("shift", False, 1, 8, 2, 2048, 64),             # D = 64: never split
    ("shift", False, 1, 8, 2, 2048, 128),
    ("symmetric_shift", True, 1, 8, 2, 640, 128),
    ("shift", False, 2, 4, 2, 384, 64),
    ("symmetric_shift", True, 8, 32, 8, 4096, 128),    # many group tasks already fill the waves
    ("shift", False, 16, 16, 4, 8192, 128),
])
def test_split_follows_the_busiest_worker(schedule, causal, B, Hq, Hkv, S, D):
    n = (S + 127) // 128
    grouped = busiest(schedule, B, Hq, Hkv, n, causal)
    split = busiest(schedule, B, Hq, Hq, n, causal)
    want = D == 128 and split * 102 < grouped * 100   # per-head partials exist at D = 128 only
    assert dash.head_split(schedule, causal, B, Hq, Hkv, S, D, P) == want


@pytest.mark.parametrize("schedule,causal,B,Hq,Hkv,S,D,window,Skv", [
    ("shift", True, 1, 32, 8, 16384, 128, 4096, None),    # causal sliding window (band tasks)
    ("shift", True, 2, 8, 2, 3000, 128, 700, None),
    ("shift", False, 1, 16, 4, 1024, 128, None, 8192),    # query and key lengths differ
    ("shift", False, 4, 8, 2, 640, 128, None, 4000),
])
def test_split_rule_with_windows_and_cross_lengths(schedule, causal, B, Hq, Hkv, S, D, window, Skv):
    n = (S + 127) // 128
    band = G.band_tiles(window) if window else None
    nkv = (Skv + 127) // 128 if Skv else None

    def load(hkv):
        tasks = G.make_tasks(schedule, B, Hq, hkv, n, causal, band, nkv)
        w = [0] * P
        for k, t in enumerate(tasks):
            w[k % P] += len(t)
        return max(w)

    want = load(Hq) * 102 < load(Hkv) * 100
    assert dash.head_split(schedule, causal, B, Hq, Hkv, S, D, P, window=window, Skv=Skv) == want


def test_llama_shape_is_split_and_ungrouped_shapes_are_not():
    assert dash.head_split("symmetric_shift", True, 1, 32, 8, 16384, 128, P)
    assert dash.head_split("auto", True, 1, 32, 8, 16384, 128, P)
    assert not dash.head_split("symmetric_shift", True, 4, 16, 16, 8192, 128, P)   # no groups
    assert not dash.head_split("descending_q", True, 1, 32, 8, 16384, 128, P)     # dynamic dispatch
    assert not dash.head_split("atomic_nondet", True, 1, 32, 8, 16384, 128, P)
    assert dash.task_heads("symmetric_shift", True, 1, 32, 8, 16384, 128, P) == 32
    assert dash.task_heads("descending_q", True, 1, 32, 8, 16384, 128, P) == 8
    assert not dash.head_split("symmetric_shift", True, 1, 32, 8, 16384, 64, P)   # D = 64


def test_rejects_bad_shapes():
    with pytest.raises(dash.DashError):
        dash.head_split("shift", False, 1, 6, 4, 512, 64, P)      # Hq % Hkv != 0
    with pytest.raises(dash.DashError):
        dash.head_split("shift", False, 1, 4, 2, 512, 64, 0)      # no workers
    with pytest.raises(dash.DashError):
        dash.head_split("shift", False, 1, 4, 2, 512, 64, P, window=128)   # window needs causal


@pytest.mark.parametrize("schedule,causal,B,Hq,Hkv,n", [
    ("shift", True, 1, 32, 32, 128),            # causal shift, dealt KV tile by KV tile
    ("shift", True, 4, 16, 16, 64),
    ("symmetric_shift", True, 1, 32, 8, 128),
    ("shift", False, 4, 16, 16, 32),
])
def test_static_makespan_without_reduction_is_the_busiest_worker(schedule, causal, B, Hq, Hkv, n):
    # with a zero reduction cost the DAG model's makespan of a static schedule is the
    # pair count of its busiest worker (tasks dealt k -> k mod P in the oracle's order)
    mk, _, _ = dash.sim_schedule(schedule, causal, B, Hq, Hkv, n, P, c=1.0, r=0.0, turn_order=False)
    assert mk == busiest(schedule, B, Hq, Hkv, n, causal)


def test_causal_shift_waves_are_balanced():
    # KV-tile-major dealing keeps the busiest of 152 workers within 4% of the mean
    tasks = G.make_tasks("shift", 1, 32, 32, 128, True)
    mean = sum(len(t) for t in tasks) / P
    assert busiest("shift", 1, 32, 32, 128, True) <= 1.04 * mean
