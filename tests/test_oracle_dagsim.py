"""Pins for the DAG schedule simulator of the oracle (no GPU).

Pinned against: the closed forms printed on the pages (golden file), the
per-SM rotation lists printed for n = 4 (golden file), the DAG lower bound,
brute force over all visit orders on tiny problems, and brute force over all
small DAGs for the zero-weight-edge lemma.
"""
import itertools
import os
import random

import numpy as np
import pytest

from oracle import dagsim as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def closed_form_rows():
    out = []
    for line in golden_rows("closed_forms.txt"):
        n, m, c, r, tc, tr, lb, sym = line.split()
        out.append((int(n), int(m), float(c), float(r), float(tc), float(tr), float(lb), float(sym)))
    return out


def makespan(sched, n, m, causal, c, r, P=None):
    s = G.build(sched, 1, m, m, n, causal, P or n)
    return G.simulate(s, c, r).makespan


@pytest.mark.parametrize("row", closed_form_rows())
def test_closed_forms(row):
    n, m, c, r, t_causal, t_rev, lb, sym = row
    # serialized ascending reaches T_causal on causal masks (and on full masks)
    assert makespan("serialized_ascending", n, m, True, c, r) == pytest.approx(t_causal)
    assert makespan("serialized_ascending", n, m, False, c, r) == pytest.approx(t_causal)
    # descending Q iteration reaches T_reversed (even m)
    assert makespan("descending_q", n, m, True, c, r) == pytest.approx(t_rev)
    # shift reaches the full-mask DAG lower bound
    assert makespan("shift", n, m, False, c, r) == pytest.approx(lb)
    # symmetric shift reaches the causal lower bound m(n+1)(c+r)/2
    assert makespan("symmetric_shift", n, m, True, c, r) == pytest.approx(sym)


@pytest.mark.parametrize("n,m", [(4, 3), (8, 5), (16, 7)])
def test_descending_odd_m_is_above_by_n_minus_1(n, m):
    # The page writes "approximately" for T_reversed; with greedy in-order
    # dispatch an odd head count lands exactly n-1 above it.
    c, r = 3.0, 1.0
    t_rev = m * (n + 1) * (c + r) / 2 + (n - 1) * r
    assert makespan("descending_q", n, m, True, c, r) == pytest.approx(t_rev + (n - 1))


def test_rotation_lists_n4():
    want = {}
    for line in golden_rows("shift_rotation_n4.txt"):
        sm, tiles = line.split(":")
        want[int(sm)] = [int(t) for t in tiles.split()]
    # the worker that owns KV tile j visits row j of the figure (whichever of
    # the P workers the dealing gives that tile to)
    s = G.build("shift", 1, 1, 1, 4, False, 4)
    seen = set()
    for cta in range(4):
        (k,) = s.cta_tasks[cta]
        j = s.tasks[k][0].j
        assert all(p.j == j for p in s.tasks[k])
        assert [p.i for p in s.tasks[k]] == want[j]
        seen.add(j)
    assert seen == {0, 1, 2, 3}


def no_waits(s, c, r):
    """True if every reduce starts right at its compute end (no bubbles)."""
    res = G.simulate(s, c, r)
    seqs = [[p for k in s.cta_tasks[cta] for p in s.tasks[k]] for cta in range(s.P)]
    for seq in seqs:
        t = 0.0
        for p in seq:
            t += c + r
            if res.reduce_end[p] != pytest.approx(t):
                return False
    return True


@pytest.mark.parametrize("n,m,P", [(4, 1, 4), (8, 3, 8), (8, 4, 5), (6, 2, 7), (16, 2, 16)])
def test_shift_full_is_conflict_free(n, m, P):
    s = G.build("shift", 1, m, m, n, False, P)
    assert no_waits(s, 3.0, 1.0)
    res = G.simulate(s, 3.0, 1.0)
    assert res.arrival == s.turn


@pytest.mark.parametrize("n,m", [(4, 2), (8, 2), (8, 4), (16, 4), (6, 2)])
def test_symmetric_shift_causal_is_conflict_free(n, m):
    s = G.build("symmetric_shift", 1, m, m, n, True, n)
    assert no_waits(s, 3.0, 1.0)


def test_visit_lists_cover_each_pair_once():
    for sched in G.SCHEDULES:
        for causal in (False, True):
            for n in (1, 2, 3, 4, 5, 8):
                s = G.build(sched, 2, 4, 2, n, causal, 3)
                pairs = [p for t in s.tasks for p in t]
                want = {(b, hq, i, j) for b in range(2) for hq in range(4) for i in range(n)
                        for j in range(n) if (not causal or j <= i)}
                assert len(pairs) == len(want)
                assert {(p.b, p.hq, p.i, p.j) for p in pairs} == want
                # a task touches one head group; symmetric tasks at most two KV tiles
                for t in s.tasks:
                    assert len({(p.b, p.hq // 2) for p in t}) == 1
                    kvs = []
                    for p in t:
                        if not kvs or kvs[-1] != p.j:
                            kvs.append(p.j)
                    assert len(kvs) == len(set(kvs)) <= 2


def test_turn_orders():
    s = G.build("serialized_ascending", 1, 2, 2, 5, True, 3)
    assert s.turn[(0, 1, 3)] == [0, 1, 2, 3]
    s = G.build("descending_q", 1, 2, 2, 5, False, 3)
    assert s.turn[(0, 0, 0)] == [0, 1, 2, 3, 4]
    assert G.build("atomic_nondet", 1, 1, 1, 4, False, 2).turn is None
    # shift with one wave: tile q receives KV q, q-1, ..., q+1 (mod n)
    s = G.build("shift", 1, 1, 1, 5, False, 5)
    for q in range(5):
        assert s.turn[(0, 0, q)] == [(q - t) % 5 for t in range(5)]


def test_symmetric_shift_full_mask_is_shift():
    a = G.build("symmetric_shift", 2, 2, 1, 6, False, 4)
    b = G.build("shift", 2, 2, 1, 6, False, 4)
    assert a.tasks == b.tasks and a.turn == b.turn


def test_brute_force_optimality_tiny():
    # Every static assignment of visit orders (one KV tile per SM, P = n,
    # accumulation order aligned with model time) is at least the chain lower
    # bound; shift attains it.  With the accumulation order fixed to ascending
    # KV index, no visit order attains it.
    n, c, r = 3, 3.0, 1.0
    lb = n * (c + r)
    shift = G.build("shift", 1, 1, 1, n, False, n)
    assert G.simulate(shift, c, r).makespan == pytest.approx(lb)
    best_aligned = best_ascending = float("inf")
    for orders in itertools.product(itertools.permutations(range(n)), repeat=n):
        s = G.build("shift", 1, 1, 1, n, False, n)
        s.tasks = [[G.Pair(0, 0, i, j) for i in orders[j]] for j in range(n)]
        aligned = {}
        for j in range(n):
            for t, i in enumerate(orders[j]):
                aligned.setdefault(i, []).append((t, j))
        s.turn = {(0, 0, i): [j for _, j in sorted(v)] for i, v in aligned.items()}
        best_aligned = min(best_aligned, G.simulate(s, c, r).makespan)
        s.turn = {(0, 0, i): list(range(n)) for i in range(n)}
        best_ascending = min(best_ascending, G.simulate(s, c, r).makespan)
    assert best_aligned == pytest.approx(lb)
    assert best_ascending > lb


def test_deadlock_detection():
    P = G.Pair
    # two SMs, each runs its own KV tile on dQ tiles 0 then 1, but the
    # accumulation orders are crossed: a cycle
    seqs = [[P(0, 0, 0, 0), P(0, 0, 1, 0)], [P(0, 0, 1, 1), P(0, 0, 0, 1)]]
    good = {P(0, 0, 0, 0): 0, P(0, 0, 0, 1): 1, P(0, 0, 1, 1): 0, P(0, 0, 1, 0): 1}
    assert G.check_tables(seqs, good)
    cyclic = {P(0, 0, 0, 0): 1, P(0, 0, 0, 1): 0, P(0, 0, 1, 1): 1, P(0, 0, 1, 0): 0}
    assert not G.check_tables(seqs, cyclic)
    missing = dict(good)
    missing[P(0, 0, 0, 1)] = 2          # rank 1 never arrives
    assert not G.check_tables(seqs, missing)


def test_lemma_brute_force():
    # Zero-weight edge lemma (gist.science DASH summary, section 2.2.B).
    # True statements: adding u->v keeps every depth iff depth(u) <= depth(v);
    # depth(u) <= depth(v) implies the critical path is unchanged.
    # The literal "iff" for the critical-path LENGTH is false (see below).
    rnd = random.Random(1234)
    cases = 0
    for N in range(2, 6):
        all_edges = [(a, b) for a in range(N) for b in range(a + 1, N)]
        for mask in range(1 << len(all_edges)):
            es = [(a, b, rnd.randint(0, 4)) for bit, (a, b) in enumerate(all_edges) if mask >> bit & 1]
            d = G.depths(N, es)
            for u in range(N):
                for v in range(N):
                    if u == v:
                        continue
                    res = G.add_zero_edge(N, es, u, v)
                    if res is None:
                        continue
                    same_depths, same_cp = res
                    cases += 1
                    assert same_depths == (d[u] <= d[v])
                    if d[u] <= d[v]:
                        assert same_cp
    assert cases > 10000


def test_lemma_iff_counterexample_for_length():
    # 3 events, edge 0->1 of weight 1; adding 1->2 (zero weight) raises
    # depth(2) from 0 to 1 although depth(1) = 1 > depth(2) = 0, yet the
    # critical path stays 1.
    es = [(0, 1, 1)]
    assert G.depths(3, es) == [0, 1, 0]
    same_depths, same_cp = G.add_zero_edge(3, es, 1, 2)
    assert not same_depths and same_cp


def test_static_turn_order_is_deadlock_free_at_any_P():
    for sched in ("shift", "symmetric_shift"):
        for causal in (False, True):
            for P in (1, 2, 3, 5, 7, 16):
                s = G.build(sched, 1, 4, 2, 6, causal, P)
                seqs = [[p for k in s.cta_tasks[c] for p in s.tasks[k]] for c in range(P)]
                assert G.check_tables(seqs, G.turn_ranks(s))


def test_band_tiles_from_element_visibility():
    """band_tiles(W) counts the tile diagonals that hold a visible element of
    a causal W-token window, checked by brute force over the elements."""
    T = 8   # a small tile makes the brute force cheap; the rule is the same for 128
    for W in range(1, 40):
        want = 0
        for t in range(0, 8):
            q = np.arange(T)[:, None] + T * t
            k = np.arange(T)[None, :]
            if ((q - k >= 0) & (q - k < W)).any():
                want = t + 1
        assert G.band_tiles(W, tile=T) == want, W
    assert G.band_tiles(1) == 1 and G.band_tiles(128) == 2 and G.band_tiles(129) == 2 and G.band_tiles(130) == 3


def test_band_wide_enough_is_causal():
    for sched in G.SCHEDULES:
        a = G.build(sched, 1, 2, 1, 6, True, 4)
        b = G.build(sched, 1, 2, 1, 6, True, 4, band=6)
        if sched == "symmetric_shift":
            continue   # with a band it is read as shift
        assert a.tasks == b.tasks
        assert a.turn == b.turn


@pytest.mark.parametrize("schedule,causal,n,band", [("shift", False, 8, None), ("symmetric_shift", True, 16, None),
                                                    ("symmetric_shift", False, 6, None), ("shift", True, 12, 4),
                                                    ("symmetric_shift", True, 9, 3)])
def test_parity_dealing_spaces_a_tiles_contributions_two_steps_apart(schedule, causal, n, band):
    # Full-mask shift, banded shift and symmetric shift deal the even tiles
    # (pairs) of every head group first, then the odd ones; with one wave per
    # parity class, the contributions a dQ tile receives from one wave are at
    # least two steps of the rotation apart (head-major dealing would give one
    # every step).
    B, H = 1, 4
    s = G.build(schedule, B, H, H, n, causal, P=10 ** 6, band=band)
    T = len(s.tasks) // (B * H)
    even = (T + 1) // 2
    for k, t in enumerate(s.tasks):
        parity = 0 if k < B * H * even else 1
        tiles = {p.j for p in t}
        if schedule == "shift" or band is not None:
            assert tiles == {(k % even) * 2 + parity if parity == 0 else ((k - B * H * even) % (T // 2)) * 2 + 1}
    for par in range(2):
        wave = [k for k in range(len(s.tasks)) if (k < B * H * even) == (par == 0)]
        times = {}
        for k in wave:
            for step, p in enumerate(s.tasks[k]):
                times.setdefault((p.b, p.hq, p.i), []).append(step)
        for tile, ts in times.items():
            ts.sort()
            assert all(b - a >= 2 for a, b in zip(ts, ts[1:])), (schedule, tile, ts)
