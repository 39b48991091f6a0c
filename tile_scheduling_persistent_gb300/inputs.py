"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws the random tensors
(Q, K, V, dO) that both the CUDA path and the CPU oracle consume, and lists
the workload shapes.  O and LSE are *derived* inputs (a forward pass) and are
produced by the caller.

Recipe: one CPU ``torch.Generator`` seeded with ``seed``; fp32 standard
normals drawn in the order Q, K, V, dO, each multiplied by its sigma and
rounded to bfloat16 (round to nearest even, torch's ``.to(torch.bfloat16)``).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

SCHEDULE_IDS = {
    "atomic_nondet": 0,
    "serialized_ascending": 1,
    "descending_q": 2,
    "shift": 3,
    "symmetric_shift": 4,
    "auto": 5,
}


@dataclass(frozen=True)
class Workload:
    name: str
    causal: bool
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    sigma_qkv: float
    sigma_do: float
    schedules: tuple
    window: int | None = None   # causal sliding window in tokens (None: none)
    Skv: int | None = None      # key/value length when it differs from S (full masks)


WORKLOADS = {
    "full_b1_h2_s512_d64": Workload(
        "full_b1_h2_s512_d64", False, 1, 2, 2, 512, 64, 1.0, 1.0,
        ("atomic_nondet", "serialized_ascending", "descending_q", "shift", "symmetric_shift")),
    "full_b4_h16_s4096_d128": Workload(
        "full_b4_h16_s4096_d128", False, 4, 16, 16, 4096, 128, 1.0, 1.0,
        ("shift", "serialized_ascending", "atomic_nondet")),
    "causal_b4_h16_s8192_d128": Workload(
        "causal_b4_h16_s8192_d128", True, 4, 16, 16, 8192, 128, 1.0, 1.0,
        ("descending_q", "symmetric_shift", "serialized_ascending", "atomic_nondet")),
    "causal_b1_h32_s16384_d64": Workload(
        "causal_b1_h32_s16384_d64", True, 1, 32, 32, 16384, 64, 1.0, 1.0,
        ("symmetric_shift", "descending_q", "shift")),   # shift: the schedule auto selects here on GB300
    "gqa_causal_b1_hq32_hkv8_s16384_d128": Workload(
        "gqa_causal_b1_hq32_hkv8_s16384_d128", True, 1, 32, 8, 16384, 128, 0.5, 1e-2,
        ("symmetric_shift", "descending_q", "shift", "serialized_ascending", "atomic_nondet")),
    # full mask at 16K: where the pages saw shift fall behind on H800 (remote-L2 latency)
    "full_b1_h16_s16384_d128": Workload(
        "full_b1_h16_s16384_d128", False, 1, 16, 16, 16384, 128, 1.0, 1.0,
        ("shift", "serialized_ascending", "descending_q", "atomic_nondet")),
    # a causal sliding window of 4096 tokens over 16K (the band mask of the
    # Ascend plan; a Mistral-style long-context layer shape)
    "window_b1_hq32_hkv8_s16384_d128_w4096": Workload(
        "window_b1_hq32_hkv8_s16384_d128_w4096", True, 1, 32, 8, 16384, 128, 0.5, 1e-2,
        ("shift", "descending_q", "serialized_ascending", "atomic_nondet"), window=4096),
    # different query and key lengths: 1K queries against 8K keys (full mask)
    "cross_b4_h16_sq1024_skv8192_d128": Workload(
        "cross_b4_h16_sq1024_skv8192_d128", False, 4, 16, 16, 1024, 128, 1.0, 1.0,
        ("shift", "serialized_ascending", "descending_q", "atomic_nondet"), Skv=8192),
}


def make_qkvdo(B: int, Hq: int, Hkv: int, S: int, D: int, seed: int = 0,
               sigma_qkv: float = 1.0, sigma_do: float = 1.0, Skv: int | None = None):
    """Seeded bf16 (q, k, v, do) on the CPU, shapes [B,H,S,D] (k, v: [B,Hkv,Skv,D])."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))

    def draw(h, sigma, L=S):
        x = torch.randn((B, h, L, D), generator=g, dtype=torch.float32)
        return (x * sigma).to(torch.bfloat16)

    q = draw(Hq, sigma_qkv)
    k = draw(Hkv, sigma_qkv, S if Skv is None else Skv)
    v = draw(Hkv, sigma_qkv, S if Skv is None else Skv)
    do = draw(Hq, sigma_do)
    return q, k, v, do


def make_workload_inputs(w: Workload, seed: int = 0):
    return make_qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed, w.sigma_qkv, w.sigma_do, w.Skv)
