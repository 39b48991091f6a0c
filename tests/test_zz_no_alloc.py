"""dash_attn_bwd_noalloc: the entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc: they have handed the device to their
own pool allocator, or run on a latency-critical path where the implicit
synchronization of cudaMalloc/cudaFree is not acceptable.  For them the
library offers dash_attn_bwd_noalloc, which takes its scratch from a fixed
device array instead of growing a workspace.  This test calls it through the
C ABI and checks that two calls in a row give the same outputs as the
regular entry point, within the tolerance the other tests use (and, for the
ordered schedules, bit for bit).  It lives in its own file so that it runs
last, and it passes alone in a fresh process as well as after the others.
It also checks the property the entry point exists for: once set up, calls
leave the device's free memory unchanged (no allocation, no workspace).
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

from tile_scheduling_persistent_gb300 import dash

from gpu_helpers import MAX_ABS, REL_L2, err, make_case, outputs, same_bits

pytestmark = pytest.mark.gpu

CASES = [((1, 2, 2, 512, 64, False), "shift"),
         ((1, 4, 2, 384, 128, True), "symmetric_shift"),
         ((2, 2, 1, 640, 64, True), "descending_q"),
         ((1, 2, 2, 256, 128, False), "atomic_nondet")]


def call_noalloc(c, sched):
    dq, dk, dv = outputs(c)
    L = dash.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = L.dash_attn_bwd_noalloc(p(c.q), p(c.k), p(c.v), p(c.o), p(c.do), p(c.lse), p(dq), p(dk), p(dv),
                                 c.B, c.Hq, c.Hkv, c.S, c.D, int(c.causal), dash._sched(sched),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == dash.OK, rc
    dqb = torch.empty(dq.shape, dtype=torch.bfloat16, device="cuda")
    dash.dq_finalize(dq, dqb)
    torch.cuda.synchronize()
    return dq, dqb, dk, dv


def call_regular(c, sched):
    # the allocation-free entry always runs one task per key/value head group
    # (it has no room for per-query-head partials): compare with that layout
    dq, dk, dv = outputs(c)
    dash.attn_bwd_debug(c.q, c.k, c.v, c.o, c.do, c.lse, dq, dk, dv, c.causal, sched, head_split=False)
    dqb = torch.empty(dq.shape, dtype=torch.bfloat16, device="cuda")
    dash.dq_finalize(dq, dqb)
    torch.cuda.synchronize()
    return dq, dqb, dk, dv


@pytest.mark.parametrize("shape,sched", CASES)
def test_noalloc_matches_regular_entry_point(shape, sched):
    c = make_case(*shape, with_ref=False)
    ref = call_regular(c, sched)
    for _ in range(2):                       # two calls in a row share the scratch
        got = call_noalloc(c, sched)
        for name, a, b in zip(("dq", "dq_bf16", "dk", "dv"), got, ref):
            rel, mx = err(a, b.float().cpu().double().numpy())
            assert rel <= REL_L2 and mx <= MAX_ABS, (name, rel, mx)
            if sched != "atomic_nondet":
                assert same_bits(a, b), name


# every ordered schedule, one full and one causal grouped-query shape: bit for
# bit the regular entry point with one task per key/value head group
ORDERED = ("serialized_ascending", "descending_q", "shift", "symmetric_shift")


@pytest.mark.parametrize("shape", [(1, 2, 2, 512, 128, False), (1, 4, 2, 384, 128, True)])
@pytest.mark.parametrize("sched", ORDERED)
def test_noalloc_bits_equal_group_task_layout(shape, sched):
    c = make_case(*shape, with_ref=False)
    ref = call_regular(c, sched)
    got = call_noalloc(c, sched)
    for name, a, b in zip(("dq", "dq_bf16", "dk", "dv"), got, ref):
        assert same_bits(a, b), (sched, name)
    code, _ = dash.get_status_noalloc()
    assert code == dash.OK


CHILD = textwrap.dedent("""
    import ctypes, sys, torch
    sys.path.insert(0, %r)
    from tile_scheduling_persistent_gb300 import dash
    from tile_scheduling_persistent_gb300.inputs import make_qkvdo
    dev = torch.device("cuda")
    B, Hq, Hkv, S, D = 1, 4, 2, 512, 128
    q, k, v, do = (t.to(dev) for t in make_qkvdo(B, Hq, Hkv, S, D, seed=3))
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, S, dtype=torch.float32, device=dev)
    dash.attn_fwd(q, k, v, o, lse, True)
    dq = torch.empty(B, Hq, S, D, dtype=torch.float32, device=dev)
    dk = torch.empty(B, Hkv, S, D, dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    torch.cuda.synchronize()
    dash.noalloc_init()
    dash.attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, True, "symmetric_shift")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for sched in ("shift", "symmetric_shift", "descending_q", "atomic_nondet"):
        dash.attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, True, sched)
        assert dash.get_status_noalloc()[0] == dash.OK
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    print("free bytes before/after", free0, free1)
    assert free1 == free0, (free0, free1)
    print("NOALLOC_OK")
""")


def test_noalloc_allocates_nothing_after_setup_fresh_process():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", CHILD % root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "NOALLOC_OK" in r.stdout, r.stdout + r.stderr


def test_noalloc_rejects_problems_beyond_its_scratch():
    c = make_case(1, 2, 2, 256, 64, False, with_ref=False)
    L = dash.lib()
    p = ctypes.c_void_p(c.q.data_ptr())
    # 512 heads of S = 16384: delta alone needs 32 MiB, more than the fixed scratch
    rc = L.dash_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 512, 512, 16384, 64, 1, 3,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == dash.ERR_SCRATCH
