"""Causal sliding window (key j visible to query i iff i - W < j <= i) on
the GPU: forward and backward parity with the fp64 oracle, the band's
accumulation orders against the simulator, bitwise reproducibility, and
W >= S giving exactly the causal results."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import dagsim as G
from tile_scheduling_persistent_gb300 import dash
from tile_scheduling_persistent_gb300.inputs import make_qkvdo

from gpu_helpers import check, same_bits

pytestmark = pytest.mark.gpu

SCHEDS = ["atomic_nondet", "serialized_ascending", "descending_q", "shift", "symmetric_shift"]
ORDERED = SCHEDS[1:]
SHAPES = {
    # name: (B, Hq, Hkv, S, D, W)
    "s512_d64_w130": (1, 2, 2, 512, 64, 130),          # n = 4, band of 3 tile diagonals
    "s640_d128_w200_gqa": (1, 4, 2, 640, 128, 200),    # n = 5, GQA 2:1
    "s700_d64_w64_gqa": (2, 2, 1, 700, 64, 64),        # ragged tail + window, B = 2
    "s1024_d128_w300": (1, 2, 2, 1024, 128, 300),      # n = 8, band of 4
    "s256_d128_w1": (1, 1, 1, 256, 128, 1),            # each query sees only its own key
}
_cases = {}


def case(name):
    if name not in _cases:
        B, Hq, Hkv, S, D, W = SHAPES[name]
        q, k, v, do = make_qkvdo(B, Hq, Hkv, S, D, seed=21)
        o, lse = A.attn_fwd(q, k, v, True, window=W)
        ref = A.attn_bwd(q, k, v, o, do, lse, True, window=W)
        dev = torch.device("cuda")
        t = {"q": q.to(dev), "k": k.to(dev), "v": v.to(dev), "do": do.to(dev),
             "o": torch.from_numpy(o).to(torch.bfloat16).to(dev), "lse": torch.from_numpy(lse).float().to(dev)}
        _cases[name] = (SHAPES[name], t, (o, lse), ref)
    return _cases[name]


def run_bwd(shape, t, sched, window, **dbg):
    B, Hq, Hkv, S, D, _ = shape
    dev = t["q"].device
    dq = torch.empty(B, Hq, S, D, dtype=torch.float32, device=dev)
    dk = torch.empty(B, Hkv, S, D, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    dash.attn_bwd(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], dq, dk, dv, True, sched, window=window)
    dqb = torch.empty(dq.shape, dtype=torch.bfloat16, device=dev)
    dash.dq_finalize(dq, dqb)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    return dq, dqb, dk, dv


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("sched", SCHEDS)
def test_window_backward_parity(name, sched):
    shape, t, _, ref = case(name)
    _, dqb, dk, dv = run_bwd(shape, t, sched, shape[5])
    for nm, got, r in (("dq", dqb, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        if not np.any(r):   # W = 1: dQ = dK = 0 exactly, a relative error has no meaning
            assert float(got.float().abs().max()) <= 1e-4, (name, sched, nm)
            continue
        check("%s %s %s" % (name, sched, nm), got, r)


@pytest.mark.parametrize("name", list(SHAPES))
def test_window_forward_parity(name):
    shape, t, (o_ref, lse_ref), _ = case(name)
    B, Hq, Hkv, S, D, W = shape
    o = torch.empty_like(t["q"])
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=o.device)
    dash.attn_fwd(t["q"], t["k"], t["v"], o, lse, True, window=W)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    check(name + " o", o, o_ref)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= 1e-4


@pytest.mark.parametrize("name", ["s512_d64_w130", "s640_d128_w200_gqa", "s700_d64_w64_gqa"])
@pytest.mark.parametrize("sched", ORDERED)
def test_window_order_log_matches_simulator_and_repeats(name, sched):
    shape, t, _, _ = case(name)
    B, Hq, Hkv, S, D, W = shape
    n = (S + 127) // 128
    band = G.band_tiles(W)
    log = torch.full((B * Hq * n, n), -1, dtype=torch.int32, device="cuda")
    dev = t["q"].device
    dq = torch.empty(B, Hq, S, D, dtype=torch.float32, device=dev)
    dk = torch.empty(B, Hkv, S, D, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    dash.attn_bwd_debug(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], dq, dk, dv, True, sched,
                        order_log=log, window=W)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    P = dash.num_ctas()
    hkv = dash.task_heads(sched, True, B, Hq, Hkv, S, D, P, window=W)
    _, turns, _ = dash.sim_schedule(sched, True, B, Hq, hkv, n, P, band=band)
    np.testing.assert_array_equal(log.cpu().numpy(), turns)   # the GPU added in the simulator's order
    for tile in range(B * Hq * n):
        i = tile % n
        assert sorted(j for j in turns[tile] if j >= 0) == list(range(max(0, i - band + 1), i + 1))
    first = run_bwd(shape, t, sched, W)
    for _ in range(4):
        again = run_bwd(shape, t, sched, W)
        for a, b in zip(first, again):
            assert same_bits(a, b), sched
    del log, dq, dk, dv


def test_window_covering_the_sequence_is_causal():
    shape, t, _, _ = case("s1024_d128_w300")
    B, Hq, Hkv, S, D, _ = shape
    for sched in ("shift", "symmetric_shift", "serialized_ascending"):
        a = run_bwd(shape, t, sched, S)
        b = run_bwd(shape, t, sched, None)
        for x, y in zip(a, b):
            assert same_bits(x, y), sched


def test_window_forward_then_backward():
    B, Hq, Hkv, S, D, W = 1, 4, 2, 640, 128, 200
    q, k, v, do = make_qkvdo(B, Hq, Hkv, S, D, seed=22)
    o_ref, lse_ref = A.attn_fwd(q, k, v, True, window=W)
    ref = A.attn_bwd(q, k, v, o_ref, do, lse_ref, True, window=W)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    dash.attn_fwd(qd, kd, vd, o, lse, True, window=W)
    dq = torch.empty(B, Hq, S, D, dtype=torch.float32, device=dev)
    dk = torch.empty(B, Hkv, S, D, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    dash.attn_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, True, "auto", window=W)
    dqb = torch.empty(dq.shape, dtype=torch.bfloat16, device=dev)
    dash.dq_finalize(dq, dqb)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    for nm, got, r in (("dq", dqb, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        check("fwd->bwd window " + nm, got, r)


def test_window_rejects_bad_arguments():
    shape, t, _, _ = case("s512_d64_w130")
    with pytest.raises(dash.DashError):
        run_bwd(shape, t, "shift", 0)
