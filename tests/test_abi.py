"""The C-ABI library loads and exports every symbol its header declares (no GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

from tile_scheduling_persistent_gb300 import dash

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols():
    src = open(os.path.join(ROOT, "include", "dash.h")).read()
    return sorted(set(re.findall(r"^\s*int\s+(dash_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(dash.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return dash.lib()


def test_every_declared_symbol_is_exported(L):
    syms = header_symbols()
    assert len(syms) >= 11
    for s in syms:
        assert hasattr(L, s), s
    assert set(syms) == set(dash.EXPORTS)


def test_argument_validation_without_a_gpu(L):
    P = ctypes.c_void_p
    ok = P(1024)            # aligned, never dereferenced (rejected before any device call)
    bad = P(1026)
    args = [ok] * 9
    # null pointer
    assert L.dash_attn_bwd(*([None] + args[1:]), 1, 2, 2, 512, 64, 0, 3, None) == dash.ERR_ARG
    # misaligned pointer
    assert L.dash_attn_bwd(*([bad] + args[1:]), 1, 2, 2, 512, 64, 0, 3, None) == dash.ERR_ARG
    # empty sequence, D unsupported, Hq % Hkv, unknown schedule, causal flag
    for (B, Hq, Hkv, S, D, causal, sched) in [(1, 2, 2, 0, 64, 0, 3), (1, 2, 2, 512, 96, 0, 3),
                                              (1, 3, 2, 512, 64, 0, 3), (1, 2, 2, 512, 64, 0, 7),
                                              (1, 2, 2, 512, 64, 2, 3), (0, 2, 2, 512, 64, 0, 3)]:
        assert L.dash_attn_bwd(*args, B, Hq, Hkv, S, D, causal, sched, None) == dash.ERR_ARG
    assert L.dash_dq_finalize(bad, ok, 16, None) == dash.ERR_ARG
    assert L.dash_attn_bwd_preprocess(ok, ok, bad, 1, 1, 128, 64, None) == dash.ERR_ARG
    assert L.dash_set_timeout_ns(10_000_000) == dash.OK
    assert L.dash_set_timeout_ns(2_000_000_000) == dash.OK


def test_simulator_rejects_bad_shapes(L):
    with pytest.raises(dash.DashError):
        dash.sim_schedule("shift", False, 1, 3, 2, 4, 4)
    assert dash.sim_check_ranks("serialized_ascending", True, 1, 1, 1, 4, 4,
                                np.zeros((4, 4), np.uint16)) == dash.ERR_ARG
