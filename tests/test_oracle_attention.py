"""Pins for the fp64 attention oracle (no GPU).

The oracle is checked against things other than itself: central finite
differences of the forward, closed-form special cases, a library autograd
routine, identities that hold for any input, and planted mistakes that each
of those checks must catch.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import attention as A


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def make(B, Hq, Hkv, S, D, seed=0, scale=1.0):
    q = rand((B, Hq, S, D), seed, scale)
    k = rand((B, Hkv, S, D), seed + 1, scale)
    v = rand((B, Hkv, S, D), seed + 2, scale)
    do = rand((B, Hq, S, D), seed + 3)
    return q, k, v, do


def loss(q, k, v, do, causal):
    o, _ = A.attn_fwd(q, k, v, causal)
    return float(np.sum(o * do))


def fd_grad(f, x, h=1e-5):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


def rel_err(a, b):
    den = max(np.linalg.norm(b), 1e-300)
    return np.linalg.norm(a - b) / den


def check_fd(B, Hq, Hkv, S, D, causal, seed=0):
    """Return the worst relative error of the oracle gradient vs finite differences."""
    q, k, v, do = make(B, Hq, Hkv, S, D, seed)
    o, lse = A.attn_fwd(q, k, v, causal)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, causal)
    f = lambda: loss(q, k, v, do, causal)  # noqa: E731
    worst = 0.0
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = fd_grad(f, x)
        if np.linalg.norm(num) < 1e-12 and np.linalg.norm(g) < 1e-12:
            continue
        worst = max(worst, rel_err(g, num))
    return worst


FD_CASES = [
    (1, 1, 1, 1, 4, False), (1, 1, 1, 3, 1, False), (1, 2, 2, 3, 4, True),
    (1, 2, 1, 8, 4, False), (1, 2, 1, 8, 4, True), (2, 1, 1, 8, 8, True),
    (1, 2, 1, 16, 8, False), (1, 2, 1, 16, 8, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", FD_CASES)
def test_finite_differences(B, Hq, Hkv, S, D, causal):
    assert check_fd(B, Hq, Hkv, S, D, causal) <= 1e-6


def test_single_key_closed_form():
    # S = 1: p = 1, O = v, ds = 0 -> dQ = dK = 0 and dV = sum of the group's dO.
    q, k, v, do = make(2, 4, 2, 1, 8, seed=5)
    for causal in (False, True):
        o, lse = A.attn_fwd(q, k, v, causal)
        dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, causal)
        assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
        want = do[:, 0::2] + do[:, 1::2]
        np.testing.assert_allclose(dv, want, rtol=0, atol=1e-14)
        np.testing.assert_allclose(o[:, 0::2], np.repeat(v, 1, axis=1), atol=1e-14)


def test_uniform_keys_closed_form():
    # All keys equal -> uniform softmax over the visible keys: O_i = mean of
    # the visible values, dQ = 0, and (full mask) dV_j = mean_i dO_i.
    B, H, S, D = 1, 2, 6, 4
    q, _, v, do = make(B, H, H, S, D, seed=7)
    k = np.broadcast_to(rand((B, H, 1, D), 9), (B, H, S, D)).copy()
    o, lse = A.attn_fwd(q, k, v, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-13)
    np.testing.assert_allclose(lse, (q @ k[:, :, :1].transpose(0, 1, 3, 2))[..., 0] / math.sqrt(D) + math.log(S),
                               atol=1e-12)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, False)
    assert np.abs(dq).max() < 1e-13
    np.testing.assert_allclose(dv, np.broadcast_to(do.mean(axis=2, keepdims=True), dv.shape), atol=1e-13)
    # causal: row i sees keys 0..i, O_i = mean(v_0..v_i)
    o, lse = A.attn_fwd(q, k, v, True)
    cm = np.cumsum(v, axis=2) / np.arange(1, S + 1)[None, None, :, None]
    np.testing.assert_allclose(o, cm, atol=1e-13)
    dq, _, _, _ = A.attn_bwd(q, k, v, o, do, lse, True)
    assert np.abs(dq).max() < 1e-13


def test_causal_first_row_and_last_key():
    # Causal: query 0 sees only key 0 -> dQ_0 = 0; key S-1 is seen only by
    # query S-1 -> dV_{S-1} = p_{S-1,S-1} dO_{S-1}.
    B, H, S, D = 1, 1, 7, 4
    q, k, v, do = make(B, H, H, S, D, seed=11)
    o, lse = A.attn_fwd(q, k, v, True)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, True)
    assert np.abs(dq[0, 0, 0]).max() < 1e-15
    s_last = q[0, 0, S - 1] @ k[0, 0, S - 1] / math.sqrt(D)
    p_last = math.exp(s_last - lse[0, 0, S - 1])
    np.testing.assert_allclose(dv[0, 0, S - 1], p_last * do[0, 0, S - 1], atol=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14)


@pytest.fixture(autouse=True, scope="module")
def _torch_one_thread():
    """The torch references here run on one thread.  Torch's multi-threaded
    fp64 CPU path was seen to return LSE values 5e-10 away from an exact
    math.fsum evaluation in about one process out of six; the single-threaded
    path and the oracle agreed with that evaluation to 1e-15."""
    threads = torch.get_num_threads()
    torch.set_num_threads(1)
    yield
    torch.set_num_threads(threads)


def torch_reference(q, k, v, do, causal):
    """fp64 torch.autograd of plain softmax attention (library routine)."""
    G = q.shape[1] // k.shape[1]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    s = tq @ kk.transpose(-1, -2) / math.sqrt(q.shape[-1])
    if causal:
        S = q.shape[2]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ vv
    lse = torch.logsumexp(s, dim=-1)
    (o * torch.tensor(do)).sum().backward()
    return o.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 33, 16), (2, 4, 2, 64, 8), (1, 4, 1, 40, 32)])
def test_matches_torch_autograd(shape, causal):
    q, k, v, do = make(*shape, seed=3)
    o_t, lse_t, dq_t, dk_t, dv_t = torch_reference(q, k, v, do, causal)
    o, lse = A.attn_fwd(q, k, v, causal)
    np.testing.assert_allclose(o, o_t, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t, rtol=1e-12, atol=1e-12)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, causal)
    for a, b in ((dq, dq_t), (dk, dk_t), (dv, dv_t)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


def test_lse_is_logsumexp_and_delta_identity():
    q, k, v, do = make(1, 2, 2, 24, 8, seed=21)
    for causal in (False, True):
        o, lse = A.attn_fwd(q, k, v, causal)
        s = q @ k.transpose(0, 1, 3, 2) / math.sqrt(8)
        if causal:
            s = np.where(np.tril(np.ones((24, 24), bool)), s, -np.inf)
        np.testing.assert_allclose(lse, scipy.special.logsumexp(s, axis=-1), atol=1e-12)
        # delta_i = <dO_i, O_i> equals sum_j p_ij dp_ij
        p = np.exp(s - lse[..., None])
        dp = do @ v.transpose(0, 1, 3, 2)
        delta = A.attn_bwd_delta(o, do)
        np.testing.assert_allclose(delta, (p * dp).sum(-1), atol=1e-12)


def test_blocking_and_sampling_agree():
    q, k, v, do = make(1, 4, 2, 96, 16, seed=31)
    for causal in (False, True):
        o, lse = A.attn_fwd(q, k, v, causal)
        o2, lse2 = A.attn_fwd(q, k, v, causal, row_block=32, workers=3)
        np.testing.assert_allclose(o, o2, atol=1e-13)
        np.testing.assert_allclose(lse, lse2, atol=1e-13)
        dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, causal)
        dq2, dk2, dv2, _ = A.attn_bwd(q, k, v, o, do, lse, causal, row_block=40, workers=2)
        for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
            np.testing.assert_allclose(a, b, atol=1e-12)
        rows = [0, 5, 63, 95]
        np.testing.assert_allclose(A.dq_rows(q, k, v, o, do, lse, causal, 0, 3, rows), dq[0, 3, rows], atol=1e-12)
        sk, sv = A.dkv_rows(q, k, v, o, do, lse, causal, 0, 1, rows)
        np.testing.assert_allclose(sk, dk[0, 1, rows], atol=1e-12)
        np.testing.assert_allclose(sv, dv[0, 1, rows], atol=1e-12)


def test_flops_nominal():
    assert A.flops_nominal(1, 2, 512, 64, False) == 10 * 512 * 512 * 64 * 2
    assert A.flops_nominal(1, 32, 16384, 128, True) == pytest.approx(5.498e12, rel=1e-3)


# ---- planted mistakes: each must be caught by the finite-difference pin ----

def _mut_no_delta(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block, window=None):
    return _orig_bwd_head(qh, kh, vh, doh, lseh, np.zeros_like(deltah), causal, scale, row_block)


def _mut_transposed_dk(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block, window=None):
    dq, dk, dv = _orig_bwd_head(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block)
    # dK built from dS (not dS^T): equivalent to swapping the roles of i and j
    s = scale * qh @ kh.T
    p = np.exp(s - lseh[:, None])
    if causal:
        p = np.where(np.tril(np.ones(p.shape, bool)), p, 0)
    ds = p * (doh @ vh.T - deltah[:, None])
    return dq, scale * ds @ qh, dv


def _mut_mask_off_by_one(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block, window=None):
    S = qh.shape[0]
    s = scale * qh @ kh.T
    p = np.exp(s - lseh[:, None])
    if causal:
        p = np.where(np.tril(np.ones((S, S), bool), -1), p, 0)   # excludes the diagonal
    dp = doh @ vh.T
    ds = p * (dp - deltah[:, None])
    return scale * ds @ kh, scale * ds.T @ qh, p.T @ doh


def _mut_sign(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block, window=None):
    dq, dk, dv = _orig_bwd_head(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block)
    return -dq, dk, dv


_orig_bwd_head = A._bwd_head


@pytest.mark.parametrize("mutant,causal", [(_mut_no_delta, False), (_mut_transposed_dk, True),
                                           (_mut_mask_off_by_one, True), (_mut_sign, False)])
def test_planted_mistakes_are_caught(monkeypatch, mutant, causal):
    monkeypatch.setattr(A, "_bwd_head", mutant)
    assert check_fd(1, 2, 1, 8, 4, causal) > 1e-3


def _mut_window_off_by_one(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block, window=None):
    # the band with one key too many (i - j <= W instead of < W)
    return _orig_bwd_head(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block,
                          None if window is None else window + 1)


def test_planted_window_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(A, "_bwd_head", _mut_window_off_by_one)
    q, k, v, do = make(1, 2, 1, 16, 8, seed=11)
    o, lse = A.attn_fwd(q, k, v, True, window=3)
    dq, _, _, _ = A.attn_bwd(q, k, v, o, do, lse, True, window=3)
    num = fd_grad(lambda: loss_w(q, k, v, do, 3), q)
    assert rel_err(dq, num) > 1e-3


# ---- the sliding window (causal band of W tokens: i - W < j <= i) ----

def loss_w(q, k, v, do, window):
    o, _ = A.attn_fwd(q, k, v, True, window=window)
    return float(np.sum(o * do))


@pytest.mark.parametrize("B,Hq,Hkv,S,D,window", [(1, 2, 1, 16, 8, 3), (2, 1, 1, 9, 4, 5), (1, 2, 2, 12, 4, 2)])
def test_window_finite_differences(B, Hq, Hkv, S, D, window):
    q, k, v, do = make(B, Hq, Hkv, S, D, seed=11)
    o, lse = A.attn_fwd(q, k, v, True, window=window)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, True, window=window)
    f = lambda: loss_w(q, k, v, do, window)  # noqa: E731
    for x, g in ((q, dq), (k, dk), (v, dv)):
        assert rel_err(g, fd_grad(f, x)) <= 1e-6


def test_window_at_least_s_is_causal():
    q, k, v, do = make(1, 2, 1, 24, 8, seed=12)
    o_c, l_c = A.attn_fwd(q, k, v, True)
    for w in (24, 25, 1000):
        o_w, l_w = A.attn_fwd(q, k, v, True, window=w)
        assert np.array_equal(o_w, o_c) and np.array_equal(l_w, l_c)
        g_c = A.attn_bwd(q, k, v, o_c, do, l_c, True)
        g_w = A.attn_bwd(q, k, v, o_w, do, l_w, True, window=w)
        for a, b in zip(g_c, g_w):
            assert np.array_equal(a, b)


def test_window_one_closed_form():
    """W = 1: every query sees only its own key, so p = 1 on the diagonal,
    O_i = v_i, LSE_i = scale <q_i, k_i>, dS = 1 * (<dO_i, v_i> - <dO_i, O_i>) = 0,
    hence dQ = dK = 0 and dV_j = the group's sum of dO_j."""
    B, Hq, Hkv, S, D = 2, 4, 2, 10, 8
    q, k, v, do = make(B, Hq, Hkv, S, D, seed=13)
    o, lse = A.attn_fwd(q, k, v, True, window=1)
    G = Hq // Hkv
    for hq in range(Hq):
        np.testing.assert_allclose(o[:, hq], v[:, hq // G], atol=1e-14)
        np.testing.assert_allclose(lse[:, hq], np.einsum("bsd,bsd->bs", q[:, hq], k[:, hq // G]) / math.sqrt(D),
                                   atol=1e-13)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, True, window=1)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    for hk in range(Hkv):
        np.testing.assert_allclose(dv[:, hk], do[:, hk * G:(hk + 1) * G].sum(axis=1), atol=1e-13)


def test_window_matches_torch_autograd_with_a_band_mask():
    q, k, v, do = make(1, 4, 2, 40, 16, seed=14)
    W, S, G = 7, 40, 2
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = tq @ tk.repeat_interleave(G, dim=1).transpose(-1, -2) / 4.0
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    s = s.masked_fill(~((j <= i) & (i - j < W)), float("-inf"))
    o_t = torch.softmax(s, dim=-1) @ tv.repeat_interleave(G, dim=1)
    (o_t * torch.tensor(do)).sum().backward()
    o, lse = A.attn_fwd(q, k, v, True, window=W)
    np.testing.assert_allclose(o, o_t.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).detach().numpy(), rtol=1e-12, atol=1e-12)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, True, window=W)
    for a, b in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-10, atol=1e-11)
    r = [0, 5, 6, 7, 39]
    np.testing.assert_allclose(A.dq_rows(q, k, v, o, do, lse, True, 0, 3, r, window=W), dq[0, 3, r], atol=1e-13)
    dk_r, dv_r = A.dkv_rows(q, k, v, o, do, lse, True, 0, 1, r, window=W)
    np.testing.assert_allclose(dk_r, dk[0, 1, r], atol=1e-13)
    np.testing.assert_allclose(dv_r, dv[0, 1, r], atol=1e-13)


def test_window_rejected_without_causal_mask():
    q, k, v, _ = make(1, 1, 1, 4, 4, seed=15)
    with pytest.raises(ValueError):
        A.attn_fwd(q, k, v, False, window=2)
    with pytest.raises(ValueError):
        A.attn_fwd(q, k, v, True, window=0)


def test_window_flops():
    assert A.flops_nominal(1, 1, 1024, 64, True, window=256) == 10.0 * 64 * (1024 * 256 - 256 * 256 / 2)
    assert A.flops_nominal(1, 1, 1024, 64, True, window=4096) == A.flops_nominal(1, 1, 1024, 64, True)


# ---- different query and key lengths (full mask) ----

def test_cross_lengths_finite_differences_and_autograd():
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 5, 9, 4
    rng = np.random.default_rng(31)
    q = rng.standard_normal((B, Hq, Sq, D))
    k = rng.standard_normal((B, Hkv, Skv, D))
    v = rng.standard_normal((B, Hkv, Skv, D))
    do = rng.standard_normal((B, Hq, Sq, D))
    o, lse = A.attn_fwd(q, k, v, False)
    dq, dk, dv, _ = A.attn_bwd(q, k, v, o, do, lse, False)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    f = lambda: loss(q, k, v, do, False)  # noqa: E731
    for x, g in ((q, dq), (k, dk), (v, dv)):
        assert rel_err(g, fd_grad(f, x)) <= 1e-6
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = tq @ tk.repeat_interleave(2, dim=1).transpose(-1, -2) / 2.0
    o_t = torch.softmax(s, dim=-1) @ tv.repeat_interleave(2, dim=1)
    (o_t * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(o, o_t.detach().numpy(), rtol=1e-12, atol=1e-12)
    for a, b in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-10, atol=1e-11)
    r = [0, 4, 8]
    dk_r, dv_r = A.dkv_rows(q, k, v, o, do, lse, False, 0, 0, r)
    np.testing.assert_allclose(dk_r, dk[0, 0, r], atol=1e-13)
    np.testing.assert_allclose(dv_r, dv[0, 0, r], atol=1e-13)
    np.testing.assert_allclose(A.dq_rows(q, k, v, o, do, lse, False, 0, 1, [0, 3]), dq[0, 1, [0, 3]], atol=1e-13)


def test_cross_lengths_need_a_full_mask():
    q, k, v, _ = make(1, 1, 1, 4, 4, seed=32)
    with pytest.raises(ValueError):
        A.attn_fwd(q, np.concatenate([k, k], axis=2), np.concatenate([v, v], axis=2), True)
