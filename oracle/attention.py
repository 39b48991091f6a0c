"""Plain fp64 softmax-attention forward and backward (the numerical oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): used by tests, the
smoke check and the CPU-baseline leg of the benchmark, never by the product.

What is computed
----------------
The DASH pages state the problem and not the equations: the backward pass
must accumulate the dQ (and dK, dV) gradients across tiles, and the order of
the dQ sum is what makes the result reproducible or not ("DASH:
Deterministic Attention Scheduling for High-Throughput", gist.science
technical summary, section 1; the Ascend FlashAttentionGrad plan on
ocdem.com, section 2.1).  The gradients themselves are those of plain
softmax attention, written out here from their textbook definition.  For
batch ``b`` and query head ``hq`` (key/value head ``hk = hq // (Hq // Hkv)``):

    s_ij  = scale * <q_i, k_j>                       scale = 1 / sqrt(D)
    allowed(i, j) = (j <= i) if causal else True      (top-left causal mask)
                    and, with a sliding window of W tokens, i - j < W
    L_i   = log sum_{j allowed} exp(s_ij)             natural log
    p_ij  = exp(s_ij - L_i)  (0 where not allowed)
    O_i   = sum_j p_ij v_j
    delta_i = <dO_i, O_i>
    dp_ij = <dO_i, v_j>
    ds_ij = p_ij * (dp_ij - delta_i)
    dQ_i  = scale * sum_j ds_ij k_j
    dK_j  = sum over the heads hq of group hk, ascending, of scale * sum_i ds_ij q_i
    dV_j  = sum over the heads hq of group hk, ascending, of sum_i p_ij dO_i

Query and key lengths may differ (``q`` [B,Hq,S_q,D], ``k``/``v`` [B,Hkv,S_kv,D]) for
the full mask, as in the Ascend plan's tiling (ocdem.com, section 2.3.1:
T_r = ceil(S1/128) query tiles, T_c = ceil(S2/128) key tiles); the causal
mask and the window need S_q = S_kv.

The sliding window (``window=W``, causal masks only) is the band mask of the
Ascend plan (ocdem.com, section 2.3.5: lower-triangular and band masks, with
tiles that are entirely masked skipped): key j is visible to query i iff
i - W < j <= i.  W >= S is the plain causal mask.

Everything is float64.  ``attn_bwd`` takes O and LSE as arguments, so the
same code gives the graded variant (exact fp64 O/LSE from ``attn_fwd``) and
the diagnostic variant (the bf16 O and fp32 LSE a GPU kernel receives).

Blocking
--------
``row_block`` (default: whole head at once) only splits the sums over query
rows into partial sums over consecutive row blocks, added in ascending block
order in fp64; it exists so that a 16384 x 16384 head does not need 2 GB per
intermediate.  Nothing else is reordered or fused.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "attn_fwd",
    "attn_bwd",
    "attn_bwd_delta",
    "dq_rows",
    "dkv_rows",
    "flops_nominal",
]


def _f64(x) -> np.ndarray:
    """Return ``x`` as a float64 numpy array (accepts torch tensors too)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def _scale(D: int, scale: float | None) -> float:
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def _check_lengths(q, k, causal: bool):
    if causal and q.shape[2] != k.shape[2]:
        raise ValueError("a causal mask needs equal query and key lengths")


def _check_window(causal: bool, window):
    if window is not None and (not causal or int(window) < 1):
        raise ValueError("a sliding window needs a causal mask and window >= 1")


def _allowed(rows: np.ndarray, S: int, causal: bool, window=None) -> np.ndarray | None:
    """Boolean mask [len(rows), S]: key j is visible to query i iff j <= i
    (and i - j < window)."""
    if not causal:
        return None
    j = np.arange(S)[None, :]
    ok = j <= rows[:, None]
    if window is not None:
        ok &= rows[:, None] - j < int(window)
    return ok


def _row_blocks(S: int, row_block: int | None):
    step = S if not row_block else int(row_block)
    for r0 in range(0, S, step):
        yield r0, min(S, r0 + step)


def _fwd_head(qh, kh, vh, causal, scale, row_block, window=None):
    S = qh.shape[0]
    O = np.empty_like(qh)
    L = np.empty(S, dtype=np.float64)
    for r0, r1 in _row_blocks(S, row_block):
        rows = np.arange(r0, r1)
        s = scale * (qh[r0:r1] @ kh.T)
        allowed = _allowed(rows, kh.shape[0], causal, window)
        if allowed is not None:
            s = np.where(allowed, s, -np.inf)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        l = e.sum(axis=1)
        L[r0:r1] = m + np.log(l)
        p = e / l[:, None]
        O[r0:r1] = p @ vh
    return O, L


def attn_fwd(q, k, v, causal: bool, scale: float | None = None,
             row_block: int | None = None, workers: int = 1, window: int | None = None):
    """Exact fp64 forward: returns (O [B,Hq,S,D], LSE [B,Hq,S])."""
    _check_window(causal, window)
    q, k, v = _f64(q), _f64(k), _f64(v)
    _check_lengths(q, k, causal)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = _scale(D, scale)
    O = np.empty_like(q)
    L = np.empty((B, Hq, S), dtype=np.float64)

    def one(bh):
        b, hq = divmod(bh, Hq)
        hk = hq // G
        O[b, hq], L[b, hq] = _fwd_head(q[b, hq], k[b, hk], v[b, hk], causal, sc, row_block, window)

    _run(one, B * Hq, workers)
    return O, L


def attn_bwd_delta(o, do) -> np.ndarray:
    """delta_i = <dO_i, O_i> (fp64), shape [B,H,S]."""
    return np.einsum("bhsd,bhsd->bhs", _f64(do), _f64(o))


def _bwd_head(qh, kh, vh, doh, lseh, deltah, causal, scale, row_block, window=None):
    S, D = qh.shape
    dq = np.empty_like(qh)
    dk = np.zeros_like(kh)
    dv = np.zeros_like(vh)
    for r0, r1 in _row_blocks(S, row_block):
        rows = np.arange(r0, r1)
        s = scale * (qh[r0:r1] @ kh.T)
        p = np.exp(s - lseh[r0:r1, None])
        allowed = _allowed(rows, kh.shape[0], causal, window)
        if allowed is not None:
            p = np.where(allowed, p, 0.0)
        dp = doh[r0:r1] @ vh.T
        ds = p * (dp - deltah[r0:r1, None])
        dq[r0:r1] = scale * (ds @ kh)
        dk += scale * (ds.T @ qh[r0:r1])
        dv += p.T @ doh[r0:r1]
    return dq, dk, dv


def attn_bwd(q, k, v, o, do, lse, causal: bool, scale: float | None = None,
             row_block: int | None = None, workers: int = 1, window: int | None = None):
    """fp64 backward.  Returns (dq, dk, dv, delta).

    ``o`` and ``lse`` are taken as given (exact from ``attn_fwd`` for the
    graded oracle, or the rounded tensors a kernel sees for the diagnostic
    one).  dK and dV of a key/value head are the sum of the per-query-head
    contributions of its group, added in ascending query-head order.
    """
    _check_window(causal, window)
    q, k, v, o, do, lse = (_f64(x) for x in (q, k, v, o, do, lse))
    _check_lengths(q, k, causal)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = _scale(D, scale)
    delta = attn_bwd_delta(o, do)
    dq = np.empty_like(q)
    Skv = k.shape[2]            # the key length may differ from the query length (full masks)
    part_k = np.empty((B, Hq, Skv, D))   # per-query-head contribution to dK / dV
    part_v = np.empty((B, Hq, Skv, D))

    def one(bh):
        b, hq = divmod(bh, Hq)
        hk = hq // G
        dq[b, hq], part_k[b, hq], part_v[b, hq] = _bwd_head(
            q[b, hq], k[b, hk], v[b, hk], do[b, hq], lse[b, hq], delta[b, hq],
            causal, sc, row_block, window)

    _run(one, B * Hq, workers)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for hq in range(Hq):            # ascending head order within each group
        dk[:, hq // G] += part_k[:, hq]
        dv[:, hq // G] += part_v[:, hq]
    return dq, dk, dv, delta


def dq_rows(q, k, v, o, do, lse, causal, b, hq, rows, scale=None, window=None):
    """dQ for selected query rows of one head, one row at a time (fp64).

    Same definition as ``attn_bwd``; cost O(S*D) per row, so it can sample
    outputs of a full-size problem.  Returns [len(rows), D].
    """
    q, k, v, o, do, lse = (_f64(x) for x in (q, k, v, o, do, lse))
    Hq, Hkv, D = q.shape[1], k.shape[1], q.shape[3]
    hk = hq // (Hq // Hkv)
    sc = _scale(D, scale)
    K, V = k[b, hk], v[b, hk]
    out = np.empty((len(rows), D))
    for n, i in enumerate(rows):
        s = sc * (K @ q[b, hq, i])
        p = np.exp(s - lse[b, hq, i])
        if causal:
            p[i + 1:] = 0.0
        if window is not None:
            p[:max(0, i - int(window) + 1)] = 0.0
        dp = V @ do[b, hq, i]
        delta = do[b, hq, i] @ o[b, hq, i]
        ds = p * (dp - delta)
        out[n] = sc * (ds @ K)
    return out


def dkv_rows(q, k, v, o, do, lse, causal, b, hk, rows, scale=None, window=None):
    """dK and dV for selected key rows of one key/value head (fp64).

    Sums the contributions of every query head of the group in ascending
    order; cost O(G*S*D) per key row.  Returns (dk [len(rows), D], dv).
    """
    q, k, v, o, do, lse = (_f64(x) for x in (q, k, v, o, do, lse))
    Hq, Hkv, S, D = q.shape[1], k.shape[1], q.shape[2], q.shape[3]
    G = Hq // Hkv
    sc = _scale(D, scale)
    dk = np.zeros((len(rows), D))
    dv = np.zeros((len(rows), D))
    for hq in range(hk * G, (hk + 1) * G):
        Q, dO = q[b, hq], do[b, hq]
        delta = np.einsum("sd,sd->s", dO, o[b, hq])
        for n, j in enumerate(rows):
            s = sc * (Q @ k[b, hk, j])
            p = np.exp(s - lse[b, hq])
            if causal:
                p[:j] = 0.0
            if window is not None:
                p[j + int(window):] = 0.0
            dp = dO @ v[b, hk, j]
            ds = p * (dp - delta)
            dk[n] += sc * (ds @ Q)
            dv[n] += p @ dO
    return dk, dv


def flops_nominal(B: int, Hq: int, S: int, D: int, causal: bool, window: int | None = None) -> float:
    """Nominal backward FLOPs: 10*D per visible (query, key) pair per query
    head, counted as S^2 (full), S^2/2 (causal) or S*W - W^2/2 (sliding
    window W <= S)."""
    if window is not None and window < S:
        return 10.0 * D * B * Hq * (S * window - window * window / 2.0)
    f = 10.0 * S * S * D * B * Hq
    return f / 2 if causal else f


def _run(fn, count: int, workers: int):
    if workers <= 1 or count <= 1:
        for i in range(count):
            fn(i)
        return
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(fn, range(count)))
