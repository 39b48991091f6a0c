"""Different query and key/value lengths (full mask) on the GPU: forward and
backward parity with the fp64 oracle, the accumulation order against the
simulator, bitwise reproducibility."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from tile_scheduling_persistent_gb300 import dash

from gpu_helpers import check, same_bits

pytestmark = pytest.mark.gpu

SCHEDS = ["atomic_nondet", "serialized_ascending", "descending_q", "shift", "symmetric_shift"]
SHAPES = {
    # name: (B, Hq, Hkv, Sq, Skv, D)
    "q256_kv640_d64": (1, 2, 2, 256, 640, 64),        # 2 query tiles, 5 key tiles
    "q640_kv256_d128_gqa": (1, 4, 2, 640, 256, 128),  # 5 query tiles, 2 key tiles
    "q200_kv333_d64_gqa": (2, 2, 1, 200, 333, 64),    # ragged tails on both sides
    "q130_kv1024_d128": (1, 1, 1, 130, 1024, 128),    # 2 query tiles (2-row tail), 8 key tiles: 4 key blocks
    "q256_kv1024_d64": (1, 2, 2, 256, 1024, 64),       # 2 query tiles, 8 key tiles: 4 key blocks
}
KEY_BLOCKS = {"q130_kv1024_d128": 4, "q256_kv1024_d64": 4}
_cases = {}


def case(name):
    if name not in _cases:
        B, Hq, Hkv, Sq, Skv, D = SHAPES[name]
        g = torch.Generator().manual_seed(41)
        f = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
        q, k, v, do = f(B, Hq, Sq, D), f(B, Hkv, Skv, D), f(B, Hkv, Skv, D), f(B, Hq, Sq, D)
        o, lse = A.attn_fwd(q, k, v, False)
        ref = A.attn_bwd(q, k, v, o, do, lse, False)
        dev = torch.device("cuda")
        t = {"q": q.to(dev), "k": k.to(dev), "v": v.to(dev), "do": do.to(dev),
             "o": torch.from_numpy(o).to(torch.bfloat16).to(dev), "lse": torch.from_numpy(lse).float().to(dev)}
        _cases[name] = (SHAPES[name], t, (o, lse), ref)
    return _cases[name]


def run_bwd(shape, t, sched, **dbg):
    B, Hq, Hkv, Sq, Skv, D = shape
    dev = t["q"].device
    dq = torch.empty(B, Hq, Sq, D, dtype=torch.float32, device=dev)
    dk = torch.empty(B, Hkv, Skv, D, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    if dbg:
        dash.attn_bwd_debug(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], dq, dk, dv, False, sched, **dbg)
    else:
        dash.attn_bwd(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], dq, dk, dv, False, sched)
    dqb = torch.empty(dq.shape, dtype=torch.bfloat16, device=dev)
    dash.dq_finalize(dq, dqb)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    return dq, dqb, dk, dv


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("sched", SCHEDS)
def test_cross_backward_parity(name, sched):
    shape, t, _, ref = case(name)
    _, dqb, dk, dv = run_bwd(shape, t, sched)
    for nm, got, r in (("dq", dqb, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        check("%s %s %s" % (name, sched, nm), got, r)


@pytest.mark.parametrize("name", list(SHAPES))
def test_cross_forward_parity(name):
    shape, t, (o_ref, lse_ref), _ = case(name)
    B, Hq, Hkv, Sq, Skv, D = shape
    o = torch.empty_like(t["q"])
    lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=o.device)
    dash.attn_fwd(t["q"], t["k"], t["v"], o, lse, False)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    check(name + " o", o, o_ref)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= 1e-4


@pytest.mark.parametrize("name", ["q256_kv640_d64", "q640_kv256_d128_gqa", "q200_kv333_d64_gqa"])
@pytest.mark.parametrize("sched", SCHEDS[1:])
def test_cross_order_log_matches_simulator_and_repeats(name, sched):
    shape, t, _, _ = case(name)
    B, Hq, Hkv, Sq, Skv, D = shape
    nq, nkv = (Sq + 127) // 128, (Skv + 127) // 128
    log = torch.full((B * Hq * nq, nkv), -1, dtype=torch.int32, device="cuda")
    first = run_bwd(shape, t, sched, order_log=log)
    P = dash.num_ctas()
    hkv = dash.task_heads(sched, False, B, Hq, Hkv, Sq, D, P, Skv=Skv)
    _, turns, _ = dash.sim_schedule(sched, False, B, Hq, hkv, nq, P, nkv=nkv)
    np.testing.assert_array_equal(log.cpu().numpy(), turns)
    for _ in range(4):
        again = run_bwd(shape, t, sched)
        for a, b in zip(first, again):
            assert same_bits(a, b), sched


def _sum_blocks(parts):
    """fp32 sum in ascending block order, each addition rounded to nearest."""
    acc = parts[0].clone()
    for p in parts[1:]:
        acc = acc + p
    return acc


@pytest.mark.parametrize("name", list(KEY_BLOCKS))
@pytest.mark.parametrize("sched", ["serialized_ascending", "descending_q"])
def test_key_blocks_equal_the_blocks_run_one_by_one(name, sched):
    """With more key tiles than query tiles the backward cuts the keys into
    blocks, runs them as extra heads of one launch and adds the blocks' dQ
    sums in ascending block order.  For the schedules whose accumulation
    order is the KV index (independent of how tasks are dealt), that equals,
    bit for bit, one call per key block followed by the same fp32 sum, with
    dK and dV the blocks' own."""
    shape, t, _, _ = case(name)
    B, Hq, Hkv, Sq, Skv, D = shape
    G = KEY_BLOCKS[name]
    whole = run_bwd(shape, t, sched)
    L = Skv // G
    dqs, dks, dvs = [], [], []
    for g in range(G):
        tb = dict(t)
        tb["k"] = t["k"][:, :, g * L:(g + 1) * L].contiguous()
        tb["v"] = t["v"][:, :, g * L:(g + 1) * L].contiguous()
        dq, _, dk, dv = run_bwd((B, Hq, Hkv, Sq, L, D), tb, sched)
        dqs.append(dq)
        dks.append(dk)
        dvs.append(dv)
    assert same_bits(whole[0], _sum_blocks(dqs))
    assert same_bits(whole[2], torch.cat(dks, dim=2))
    assert same_bits(whole[3], torch.cat(dvs, dim=2))


@pytest.mark.parametrize("name", list(KEY_BLOCKS))
@pytest.mark.parametrize("sched", SCHEDS[1:])
def test_key_blocks_repeat_bitwise(name, sched):
    shape, t, _, _ = case(name)
    first = run_bwd(shape, t, sched)
    for _ in range(4):
        again = run_bwd(shape, t, sched)
        for a, b in zip(first, again):
            assert same_bits(a, b), sched
