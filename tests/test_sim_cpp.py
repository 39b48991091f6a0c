"""The product's C++ schedule simulator agrees with the oracle's Python one (no GPU).

Makespans, accumulation orders and deadlock verdicts must be identical; the
two implementations share no code.
"""
import os

import numpy as np
import pytest

from oracle import dagsim as G
from tile_scheduling_persistent_gb300 import dash
from tile_scheduling_persistent_gb300.inputs import WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not os.path.exists(dash.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    dash.lib()


def oracle_turns(s, B, Hq, n):
    out = np.full((B * Hq * n, n), -1, np.int32)
    for (b, hq, i), js in s.turn.items():
        out[(b * Hq + hq) * n + i, :len(js)] = js
    return out


CASES = [(sched, causal, B, Hq, Hkv, n, P)
         for sched in G.SCHEDULES
         for causal in (False, True)
         for (B, Hq, Hkv, n, P) in [(1, 1, 1, 4, 4), (1, 2, 2, 5, 3), (2, 4, 2, 6, 5), (1, 4, 1, 8, 7),
                                    (1, 3, 3, 7, 16), (2, 2, 2, 4, 1)]]


@pytest.mark.parametrize("sched,causal,B,Hq,Hkv,n,P", CASES)
def test_cpp_matches_oracle(sched, causal, B, Hq, Hkv, n, P):
    for c, r in ((3.0, 1.0), (1.0, 2.5)):
        s = G.build(sched, B, Hq, Hkv, n, causal, P)
        want = G.simulate(s, c, r)
        mk, turns, ntasks = dash.sim_schedule(sched, causal, B, Hq, Hkv, n, P, c, r)
        assert ntasks == len(s.tasks)
        assert mk == pytest.approx(want.makespan)
        if s.turn is not None:
            np.testing.assert_array_equal(turns, oracle_turns(s, B, Hq, n))
        else:
            want_arrival = np.full_like(turns, -1)
            for (b, hq, i), js in want.arrival.items():
                want_arrival[(b * Hq + hq) * n + i, :len(js)] = js
            np.testing.assert_array_equal(turns, want_arrival)


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("P", [148, 152])
def test_cpp_matches_oracle_at_workload_shapes(name, P):
    w = WORKLOADS[name]
    n = w.S // 128
    if w.B * w.Hq * n * n > 300_000 and P == 148:
        pytest.skip("one SM count is enough for the largest shapes")
    for sched in w.schedules:
        if sched == "atomic_nondet":
            continue
        band = G.band_tiles(w.window) if w.window else None
        nkv = (w.Skv + 127) // 128 if w.Skv else None
        s = G.build(sched, w.B, w.Hq, w.Hkv, n, w.causal, P, band=band, nkv=nkv)
        _, turns, ntasks = dash.sim_schedule(sched, w.causal, w.B, w.Hq, w.Hkv, n, P, 1.0, 1.0, band=band,
                                             nkv=nkv)
        assert ntasks == len(s.tasks)
        want = np.full(turns.shape, -1, np.int32)
        for (b, hq, i), js in s.turn.items():
            want[(b * w.Hq + hq) * n + i, :len(js)] = js
        np.testing.assert_array_equal(turns, want)


def ranks_from_turns(turns, n):
    ranks = np.full(turns.shape, 0xFFFF, np.uint16)
    for t in range(turns.shape[0]):
        for r, j in enumerate(turns[t]):
            if j >= 0:
                ranks[t, j] = r
    return ranks


@pytest.mark.parametrize("causal", [False, True])
def test_check_ranks(causal):
    B, Hq, Hkv, n, P = 1, 2, 1, 6, 4
    for sched in ("shift", "symmetric_shift"):
        _, turns, _ = dash.sim_schedule(sched, causal, B, Hq, Hkv, n, P)
        ranks = ranks_from_turns(turns, n)
        assert dash.sim_check_ranks(sched, causal, B, Hq, Hkv, n, P, ranks) == dash.OK
        # missing predecessor: rank 1 of tile 5 replaced by 2 (duplicate 2)
        bad = ranks.copy()
        t = 5
        j1 = int(turns[t, 1])
        bad[t, j1] = 2
        assert dash.sim_check_ranks(sched, causal, B, Hq, Hkv, n, P, bad) == dash.ERR_DEADLOCK
        # reversed order on every tile: valid permutation, but it must cycle
        rev = ranks.copy()
        for tt in range(turns.shape[0]):
            js = [j for j in turns[tt] if j >= 0]
            for r, j in enumerate(reversed(js)):
                rev[tt, j] = r
        verdict = dash.sim_check_ranks(sched, causal, B, Hq, Hkv, n, P, rev)
        seqs_model = G.build(sched, B, Hq, Hkv, n, causal, P)
        seqs = [[p for k in seqs_model.cta_tasks[c] for p in seqs_model.tasks[k]] for c in range(P)]
        pr = {p: int(rev[(p.b * Hq + p.hq) * n + p.i, p.j]) for t in seqs_model.tasks for p in t}
        assert (verdict == dash.OK) == G.check_tables(seqs, pr)


BAND_CASES = [(sched, B, Hq, Hkv, n, band, P)
              for sched in G.SCHEDULES
              for (B, Hq, Hkv, n, band, P) in [(1, 1, 1, 6, 1, 4), (1, 2, 2, 7, 2, 3), (2, 4, 2, 8, 3, 5),
                                               (1, 4, 1, 9, 4, 7), (1, 2, 1, 5, 9, 16), (2, 2, 2, 6, 6, 1)]]


@pytest.mark.parametrize("sched,B,Hq,Hkv,n,band,P", BAND_CASES)
def test_cpp_matches_oracle_with_a_band(sched, B, Hq, Hkv, n, band, P):
    """A causal sliding window: tiles outside the band are skipped in both
    simulators; turn orders and makespans agree."""
    for c, r in ((3.0, 1.0), (1.0, 2.5)):
        s = G.build(sched, B, Hq, Hkv, n, True, P, band=band)
        want = G.simulate(s, c, r)
        mk, turns, ntasks = dash.sim_schedule(sched, True, B, Hq, Hkv, n, P, c, r, band=band)
        assert ntasks == len(s.tasks)
        assert mk == pytest.approx(want.makespan)
        if s.turn is not None:
            np.testing.assert_array_equal(turns, oracle_turns(s, B, Hq, n))
        # every dQ tile receives exactly the KV tiles of its band
        for t in range(B * Hq * n):
            i = t % n
            got = sorted(j for j in turns[t] if j >= 0)
            assert got == list(range(max(0, i - band + 1), i + 1))


CROSS_CASES = [(sched, B, Hq, Hkv, nq, nkv, P)
               for sched in G.SCHEDULES
               for (B, Hq, Hkv, nq, nkv, P) in [(1, 1, 1, 3, 7, 4), (1, 2, 2, 6, 2, 3), (2, 4, 2, 5, 9, 5),
                                                (1, 2, 1, 1, 4, 16), (1, 3, 3, 8, 1, 2)]]


@pytest.mark.parametrize("sched,B,Hq,Hkv,nq,nkv,P", CROSS_CASES)
def test_cpp_matches_oracle_with_different_lengths(sched, B, Hq, Hkv, nq, nkv, P):
    """Full mask, nq query tiles and nkv key/value tiles: both simulators give
    the same makespans and turn orders, and every dQ tile receives every KV tile."""
    for c, r in ((3.0, 1.0), (1.0, 2.5)):
        s = G.build(sched, B, Hq, Hkv, nq, False, P, nkv=nkv)
        want = G.simulate(s, c, r)
        mk, turns, ntasks = dash.sim_schedule(sched, False, B, Hq, Hkv, nq, P, c, r, nkv=nkv)
        assert turns.shape == (B * Hq * nq, nkv)
        assert ntasks == len(s.tasks) == B * Hkv * nkv
        assert mk == pytest.approx(want.makespan)
        if s.turn is not None:
            out = np.full((B * Hq * nq, nkv), -1, np.int32)
            for (b, hq, i), js in s.turn.items():
                out[(b * Hq + hq) * nq + i, :len(js)] = js
            np.testing.assert_array_equal(turns, out)
            for row in turns:
                assert sorted(row) == list(range(nkv))
