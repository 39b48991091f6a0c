"""Single-tile probe: each tcgen05 product of the kernel, checked on its own.

The probe runs one (KV tile, Q tile) pair through the same device building
blocks as the persistent kernel (TMA swizzled boxes, K-major and MN-major
shared-memory descriptors, the tensor-memory A operand, the softmax and dS
warps) and dumps every intermediate.  Each is compared with a plain fp64
matrix product of the same bf16 operands, so a wrong descriptor field, a
transposed operand or a swizzle mismatch shows up in the product it affects.
"""
import math

import numpy as np
import pytest
import torch

from tile_scheduling_persistent_gb300 import dash

pytestmark = pytest.mark.gpu


def bf16_round(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("diag", [False, True])
def test_tile_probe(D, diag):
    g = torch.Generator().manual_seed(100 + D + diag)
    k, v, q, do = (torch.randn(128, D, generator=g).to(torch.bfloat16) for _ in range(4))
    K, V, Q, dO = (x.double().numpy() for x in (k, v, q, do))
    scale = 1.0 / math.sqrt(D)
    s = Q @ K.T * scale                                   # [q, kv]
    if diag:
        s = np.where(np.tril(np.ones((128, 128), bool)), s, -np.inf)
    lse = np.log(np.exp(s - s.max(1, keepdims=True)).sum(1)) + s.max(1)
    delta = torch.randn(128, generator=g).double().numpy() * 0.1
    lse32 = lse.astype(np.float32)
    delta32 = delta.astype(np.float32)
    dev = torch.device("cuda")
    out = dash.tile_probe(k.to(dev), v.to(dev), q.to(dev), do.to(dev),
                          torch.from_numpy(lse32).to(dev), torch.from_numpy(delta32).to(dev), diag=diag)
    got = {n: t.double().cpu().numpy() for n, t in out.items()}

    # S^T = K Q^T (fp32 accumulation of bf16 products)
    sT = K @ Q.T
    np.testing.assert_allclose(got["sT"], sT, rtol=0, atol=1e-4 * np.abs(sT).max())
    # P^T = exp(scale S^T - LSE[q]), masked where kv > q on a diagonal tile
    pT = np.exp(scale * sT - lse32.astype(np.float64)[None, :])
    if diag:
        pT = np.where(np.triu(np.ones((128, 128), bool)), pT, 0.0)
    np.testing.assert_allclose(got["pT"], pT, rtol=1e-4, atol=1e-7)
    # dP^T = V dO^T
    dpT = V @ dO.T
    np.testing.assert_allclose(got["dpT"], dpT, rtol=0, atol=1e-4 * np.abs(dpT).max())
    # dS^T = bf16(scale * P^T o (dP^T - delta[q]))  (from the kernel's own P and dP)
    dsT = scale * got["pT"] * (got["dpT"] - delta32.astype(np.float64)[None, :])
    np.testing.assert_allclose(got["dsT"], bf16_round(dsT), rtol=8e-3, atol=1e-6 * np.abs(dsT).max())
    # dV = bf16(P^T) dO   (A operand from tensor memory)
    pT_b = bf16_round(got["pT"])
    dv = pT_b @ dO
    np.testing.assert_allclose(got["dv"], dv, rtol=0, atol=1e-4 * np.abs(dv).max() + 1e-6)
    # dK = dS^T Q   (B operand MN-major)
    dk = got["dsT"] @ Q
    np.testing.assert_allclose(got["dk"], dk, rtol=0, atol=1e-4 * np.abs(dk).max() + 1e-7)
    # dQ = dS K = (dS^T)^T K   (A and B operands MN-major)
    dq = got["dsT"].T @ K
    np.testing.assert_allclose(got["dq"], dq, rtol=0, atol=1e-4 * np.abs(dq).max() + 1e-7)
