"""Shared set-up for the GPU tests: seeded inputs, oracle references, checks."""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from oracle import attention as A
from tile_scheduling_persistent_gb300 import dash
from tile_scheduling_persistent_gb300.inputs import make_qkvdo

# Tolerances on bf16 outputs vs the fp64 oracle (whole tensor).
REL_L2 = 5e-3
MAX_ABS = 2e-2


@dataclass
class Case:
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    causal: bool
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    o: torch.Tensor
    do: torch.Tensor
    lse: torch.Tensor
    ref: tuple | None = None      # (dq, dk, dv, delta) fp64

    @property
    def n(self):
        return (self.S + 127) // 128   # the last tile may be partial


def make_case(B, Hq, Hkv, S, D, causal, seed=0, sigma_qkv=1.0, sigma_do=1.0, with_ref=True):
    q, k, v, do = make_qkvdo(B, Hq, Hkv, S, D, seed, sigma_qkv, sigma_do)
    o, lse = A.attn_fwd(q, k, v, causal)
    ref = A.attn_bwd(q, k, v, o, do, lse, causal) if with_ref else None
    dev = torch.device("cuda")
    return Case(B, Hq, Hkv, S, D, causal, q.to(dev), k.to(dev), v.to(dev),
                torch.from_numpy(o).to(torch.bfloat16).to(dev), do.to(dev),
                torch.from_numpy(lse).to(torch.float32).to(dev), ref)


def outputs(c: Case):
    dev = c.q.device
    dq = torch.empty(c.B, c.Hq, c.S, c.D, dtype=torch.float32, device=dev)
    dk = torch.empty(c.B, c.Hkv, c.S, c.D, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    return dq, dk, dv


def run(c: Case, sched, stream=None, **dbg):
    dq, dk, dv = outputs(c)
    if dbg:
        dash.attn_bwd_debug(c.q, c.k, c.v, c.o, c.do, c.lse, dq, dk, dv, c.causal, sched, stream=stream, **dbg)
    else:
        dash.attn_bwd(c.q, c.k, c.v, c.o, c.do, c.lse, dq, dk, dv, c.causal, sched, stream=stream)
    dqb = torch.empty(dq.shape, dtype=torch.bfloat16, device=dq.device)
    dash.dq_finalize(dq, dqb, stream=stream)
    code, info = dash.get_status(stream)
    assert code == 0, "device status %d %s" % (code, info)
    return dq, dqb, dk, dv


def err(got, ref):
    g = got.float().cpu().numpy().astype(np.float64) if isinstance(got, torch.Tensor) else got
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300)
    return rel, float(np.abs(g - ref).max())


def check(name, got, ref, rel_tol=REL_L2, abs_tol=MAX_ABS):
    rel, mx = err(got, ref)
    assert rel <= rel_tol and mx <= abs_tol, "%s: rel_L2 %.3e (<= %.1e), max_abs %.3e (<= %.1e)" % (
        name, rel, rel_tol, mx, abs_tol)
    return rel, mx


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def sim_turns(c: Case, sched):
    """The simulator's accumulation order for the backward of case c (with
    grouped-query heads split per query head when the library does)."""
    P = dash.num_ctas()
    hkv = dash.task_heads(sched, c.causal, c.B, c.Hq, c.Hkv, c.S, c.D, P)
    _, turns, _ = dash.sim_schedule(sched, c.causal, c.B, c.Hq, hkv, c.n, P)
    return turns


def gpu_forward_fp32(q, k, v, causal, rows=2048):
    """Plain PyTorch fp32 forward on the GPU (input synthesis for large shapes)."""
    B, Hq, S, D = q.shape
    G = Hq // k.shape[1]
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        for h in range(Hq):
            K = k[b, h // G].float()
            V = v[b, h // G].float()
            for r0 in range(0, S, rows):
                s = (q[b, h, r0:r0 + rows].float() @ K.T) * scale
                if causal:
                    idx = torch.arange(r0, min(S, r0 + rows), device=q.device)
                    s.masked_fill_(torch.arange(S, device=q.device)[None, :] > idx[:, None], float("-inf"))
                l = torch.logsumexp(s, dim=-1)
                lse[b, h, r0:r0 + rows] = l
                o[b, h, r0:r0 + rows] = (torch.exp(s - l[:, None]) @ V).to(torch.bfloat16)
    return o, lse
