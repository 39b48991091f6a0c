"""Grouped-query heads run as one task per query head (dK/dV summed over the
group afterwards in ascending head order) or as one task per key/value head
group: both agree with the fp64 oracle, each is bitwise reproducible, and
each adds dQ in the simulator's order for its own task structure."""
import numpy as np
import pytest
import torch

from tile_scheduling_persistent_gb300 import dash

from gpu_helpers import check, make_case, run, same_bits

pytestmark = pytest.mark.gpu

SHAPES = {
    # name: (B, Hq, Hkv, S, D, causal, schedule)
    "causal_s640_d128_g4_sym": (1, 8, 2, 640, 128, True, "symmetric_shift"),
    "full_s384_d128_g2_shift": (2, 4, 2, 384, 128, False, "shift"),
    "causal_s333_d128_g3_shift": (1, 6, 2, 333, 128, True, "shift"),   # ragged tail
}
_cases = {}


def case(name):
    if name not in _cases:
        B, Hq, Hkv, S, D, causal, _ = SHAPES[name]
        _cases[name] = make_case(B, Hq, Hkv, S, D, causal, seed=7)
    return _cases[name]


@pytest.mark.parametrize("split", [True, False])
@pytest.mark.parametrize("name", list(SHAPES))
def test_split_and_grouped_tasks(name, split):
    B, Hq, Hkv, S, D, causal, sched = SHAPES[name]
    c = case(name)
    n = (S + 127) // 128
    log = torch.full((B * Hq * n, n), -1, dtype=torch.int32, device="cuda")
    dq, dqb, dk, dv = run(c, sched, order_log=log, head_split=split)
    for nm, got, ref in (("dq", dqb, c.ref[0]), ("dk", dk, c.ref[1]), ("dv", dv, c.ref[2])):
        check("%s split=%s %s" % (name, split, nm), got, ref)
    # the order: that of Hkv = Hq (one task per query head) or of the real Hkv
    _, turns, _ = dash.sim_schedule(sched, causal, B, Hq, Hq if split else Hkv, n, dash.num_ctas())
    np.testing.assert_array_equal(log.cpu().numpy(), turns)
    for _ in range(3):
        again = run(c, sched, head_split=split)
        for a, b in zip((dq, dqb, dk, dv), again):
            assert same_bits(a, b)


def test_library_choice_is_one_of_the_two():
    # with no override the library runs what dash_head_split names
    name = "causal_s640_d128_g4_sym"
    B, Hq, Hkv, S, D, causal, sched = SHAPES[name]
    c = case(name)
    chosen = dash.head_split(sched, causal, B, Hq, Hkv, S, D, dash.num_ctas())
    auto = run(c, sched)
    forced = run(c, sched, head_split=chosen)
    for a, b in zip(auto, forced):
        assert same_bits(a, b)

