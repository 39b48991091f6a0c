"""GPU forward pass (O, LSE): parity with the fp64 oracle, reproducibility,
and a forward -> backward step that uses only this library on the GPU."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from tile_scheduling_persistent_gb300 import dash
from tile_scheduling_persistent_gb300.inputs import make_qkvdo

from gpu_helpers import check, same_bits

pytestmark = pytest.mark.gpu

SHAPES = {
    # name: (B, Hq, Hkv, S, D, causal)
    "full_s512_d64": (1, 2, 2, 512, 64, False),
    "causal_s512_d64": (1, 2, 2, 512, 64, True),
    "full_s384_d128_gqa": (1, 4, 2, 384, 128, False),
    "causal_s384_d128_gqa": (1, 4, 2, 384, 128, True),
    "causal_s640_d64_gqa": (2, 2, 1, 640, 64, True),
    "causal_s1024_d128": (1, 3, 3, 1024, 128, True),
    "causal_s128_d64": (1, 1, 1, 128, 64, True),
    "full_s128_d128": (1, 1, 1, 128, 128, False),
    # ragged lengths: the last tile is partial (S % 128 != 0)
    "full_s200_d64": (1, 2, 2, 200, 64, False),
    "causal_s333_d128_gqa": (1, 4, 2, 333, 128, True),
    "full_s130_d128": (1, 1, 1, 130, 128, False),
    "causal_s100_d64": (1, 1, 1, 100, 64, True),
}
# More than twice as many Q tiles (CTAs) as a GB300 has SMs, so the grid runs
# in several waves (uneven tile lengths on causal masks, a ragged tail, a
# window), each against the oracle and repeated bit for bit.
MANY = {
    # name: (B, Hq, Hkv, S, D, causal, window)
    "full_b2_h16_s1280_d64": (2, 16, 16, 1280, 64, False, None),
    "causal_b2_h16_s1280_d128_gqa": (2, 16, 4, 1280, 128, True, None),
    "causal_b2_h16_s1200_d64_gqa_ragged": (2, 16, 8, 1200, 64, True, None),
    "window_b2_h16_s1280_d128_w300": (2, 16, 16, 1280, 128, True, 300),
}
LSE_ABS = 1e-4   # fp32 LSE of O(10): the kernel's fp32 score sums against the exact fp64 value


def forward(q, k, v, causal):
    B, Hq, S, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device)
    dash.attn_fwd(q, k, v, o, lse, causal)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    return o, lse


@pytest.mark.parametrize("name", list(SHAPES))
def test_forward_parity(name):
    B, Hq, Hkv, S, D, causal = SHAPES[name]
    q, k, v, _ = make_qkvdo(B, Hq, Hkv, S, D, seed=3)
    o_ref, lse_ref = A.attn_fwd(q, k, v, causal)
    dev = torch.device("cuda")
    o, lse = forward(q.to(dev), k.to(dev), v.to(dev), causal)
    check(name + " o", o, o_ref)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= LSE_ABS


@pytest.mark.parametrize("name", list(MANY))
def test_forward_parity_many_tiles(name):
    B, Hq, Hkv, S, D, causal, window = MANY[name]
    assert B * Hq * ((S + 127) // 128) > 2 * 152
    q, k, v, _ = make_qkvdo(B, Hq, Hkv, S, D, seed=8)
    o_ref, lse_ref = A.attn_fwd(q, k, v, causal, window=window)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    dash.attn_fwd(q, k, v, o, lse, causal, window=window)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    check(name + " o", o, o_ref)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= LSE_ABS
    o2 = torch.empty_like(o)
    lse2 = torch.empty_like(lse)
    dash.attn_fwd(q, k, v, o2, lse2, causal, window=window)
    assert same_bits(o, o2) and same_bits(lse, lse2)


def test_forward_rescaling_many_tiles():
    # sigma 3 scores (frequent in-loop rescaling of O) with 320 Q tiles
    B, Hq, Hkv, S, D, causal = 2, 16, 16, 1280, 64, False
    q, k, _, _ = make_qkvdo(B, Hq, Hkv, S, D, seed=5, sigma_qkv=3.0)
    _, _, v, _ = make_qkvdo(B, Hq, Hkv, S, D, seed=7)
    o_ref, lse_ref = A.attn_fwd(q, k, v, causal)
    dev = torch.device("cuda")
    o, lse = forward(q.to(dev), k.to(dev), v.to(dev), causal)
    check("o", o, o_ref)
    rel = np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref) / np.maximum(np.abs(lse_ref), 1.0)
    assert rel.max() <= 1e-5


def test_forward_large_scores_need_rescaling():
    # sigma 3 inputs: row maxima grow by far more than 2^8 from tile to tile,
    # so the running maximum is raised and O rescaled inside the loop
    B, Hq, Hkv, S, D, causal = 1, 2, 2, 1024, 64, False
    q, k, _, _ = make_qkvdo(B, Hq, Hkv, S, D, seed=5, sigma_qkv=3.0)
    _, _, v, _ = make_qkvdo(B, Hq, Hkv, S, D, seed=7)   # |O| stays where bf16 rounding meets max-abs
    o_ref, lse_ref = A.attn_fwd(q, k, v, causal)
    dev = torch.device("cuda")
    o, lse = forward(q.to(dev), k.to(dev), v.to(dev), causal)
    check("o", o, o_ref)
    rel = np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref) / np.maximum(np.abs(lse_ref), 1.0)
    assert rel.max() <= 1e-5


def test_forward_bitwise_reproducible():
    B, Hq, Hkv, S, D, causal = SHAPES["causal_s1024_d128"]
    q, k, v, _ = make_qkvdo(B, Hq, Hkv, S, D, seed=4)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    first = forward(q, k, v, causal)
    for _ in range(5):
        again = forward(q, k, v, causal)
        assert same_bits(first[0], again[0]) and same_bits(first[1], again[1])


@pytest.mark.parametrize("name,sched", [("causal_s384_d128_gqa", "symmetric_shift"),
                                        ("full_s512_d64", "shift"), ("causal_s640_d64_gqa", "auto"),
                                        ("causal_s333_d128_gqa", "shift"), ("full_s200_d64", "descending_q")])
def test_forward_then_backward_on_the_gpu(name, sched):
    """A whole training step's attention on the GPU (forward, then the
    deterministic backward on the forward's own O and LSE) against the exact
    fp64 oracle."""
    B, Hq, Hkv, S, D, causal = SHAPES[name]
    q, k, v, do = make_qkvdo(B, Hq, Hkv, S, D, seed=6)
    o_ref, lse_ref = A.attn_fwd(q, k, v, causal)
    ref = A.attn_bwd(q, k, v, o_ref, do, lse_ref, causal)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = forward(qd, kd, vd, causal)
    dq = torch.empty(B, Hq, S, D, dtype=torch.float32, device=dev)
    dk = torch.empty(B, Hkv, S, D, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    dash.attn_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, causal, sched)
    dqb = torch.empty(dq.shape, dtype=torch.bfloat16, device=dev)
    dash.dq_finalize(dq, dqb)
    code, info = dash.get_status()
    assert code == 0, (code, info)
    for nm, got, r in (("dq", dqb, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        check(name + " " + nm, got, r)


def test_forward_rejects_bad_shapes():
    dev = torch.device("cuda")
    q = torch.zeros(1, 2, 256, 96, dtype=torch.bfloat16, device=dev)   # D = 96 is not supported
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 256, dtype=torch.float32, device=dev)
    with pytest.raises(dash.DashError):
        dash.attn_fwd(q, q, q, o, lse, False)
