"""DAG model of the deterministic attention backward and its tile schedules.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The model (DASH technical summary on gist.science, section 2.1; the pwwt.cn
write-up, section 2.2 "computation-graph modelling layer"):

* the work is a set of *pairs* (KV tile j, Q tile i) of one query head; each
  pair is a compute node of cost ``c`` followed by a reduce node of cost
  ``r`` that adds the pair's dQ partial into dQ tile i;
* all pairs of one KV tile (a *task*) run back to back on one SM, so each SM
  is a chain compute -> reduce -> compute -> reduce ... (the summary's
  "operations for one KV tile execute contiguously on one SM");
* the reduces into one dQ tile happen in a fixed order (the accumulation
  order); the reduce of the k-th contributor may start only after the
  (k-1)-th has finished (a zero-weight edge from the predecessor's reduce
  end to the successor's reduce start);
* the objective is the critical-path length (makespan).

Schedules (summary section 2.2; write-up section 2.3):

``serialized_ascending``
    Q tiles visited in ascending order; accumulation order = ascending KV
    index (the FlashAttention-3 style deterministic baseline).
``descending_q``
    Q tiles visited in descending order; the accumulation order is still
    ascending KV index.
``shift``
    The SM owning KV tile j visits Q tiles j, j+1, ..., n-1, 0, ..., j-1
    (the summary's cyclic order "SM i processes i, i+1, ..., N-1, 0, ...,
    i-1", read with the KV tile resident and the Q tiles rotating); on a
    causal mask the masked tiles are skipped.
``symmetric_shift``
    Causal masks: KV tiles jp and n-1-jp form one task.  Phase 1 (the dense
    rectangle): KV jp visits the last h = n//2 Q tiles in rotated order
    (n-h) + ((jp + t) mod h).  Phase 2 (the folded triangle): KV jp visits Q
    jp .. n-h-1 ascending, then KV n-1-jp visits Q n-1 .. n-1-jp descending.
    Odd n: the middle tile forms a task of its own (descending visits).  On a
    full mask this schedule is ``shift``.
``atomic_nondet``
    Ascending visits, no accumulation order (no reduce edges).

Assignment: the static schedules (shift, symmetric shift) give task k to SM
``k mod P``; the others use greedy in-order dispatch (the next task goes to
the SM that becomes free first, lowest SM id on ties).  For the static
schedules the accumulation order of a dQ tile is ascending *model time*
(the position of the pair in its SM's unit-step sequence), ties broken by
lower KV index: the order in which the reductions arrive when every pair
takes the same time, i.e. the accumulation order aligned with the execution
schedule.

Task order: head group by head group (b, hk, then the KV tile), except causal
shift without a window, whose tasks are taken KV tile by KV tile (all groups'
tile 0, then tile 1, ...), which balances the round-robin waves when tile j
has n - j pairs (a GB300 choice; the pages leave the enumeration open).

GQA: a task is one KV tile of head group hk; it runs the pairs of every query
head of the group, ascending, each head's visits in the schedule's order
(for symmetric shift: all heads' phase 1 + phase 2a of KV jp, then all
heads' phase 2b of KV n-1-jp).
"""
from __future__ import annotations

from collections import defaultdict, deque
from dataclasses import dataclass, field

SCHEDULES = ("atomic_nondet", "serialized_ascending", "descending_q", "shift",
             "symmetric_shift")
STATIC = ("shift", "symmetric_shift")


@dataclass(frozen=True)
class Pair:
    """One unit of work: dQ tile (b, hq, i) receives the partial of KV tile j."""
    b: int
    hq: int
    i: int      # Q tile
    j: int      # KV tile


@dataclass
class Schedule:
    name: str
    B: int
    Hq: int
    Hkv: int
    n: int
    causal: bool
    P: int
    tasks: list                      # list[list[Pair]] in dispatch order
    static: bool
    cta_tasks: list | None = None    # static: per SM, its task indices in order
    turn: dict | None = None         # dQ tile (b, hq, i) -> KV indices in order


@dataclass
class SimResult:
    makespan: float
    cta_of_task: list
    reduce_end: dict = field(default_factory=dict)  # Pair -> reduce end time
    arrival: dict = field(default_factory=dict)     # dQ tile -> KV order by time


# --------------------------------------------------------------------------
# visit lists
# --------------------------------------------------------------------------

def band_tiles(window: int, tile: int = 128) -> int:
    """Number of tile diagonals a causal sliding window of `window` tokens
    touches: tile pair (i, j) holds a visible (query, key) element iff
    0 <= i - j < band_tiles(window).  Diagonal t >= 1 holds one iff its
    smallest query-key distance, tile * t - (tile - 1), is below the window."""
    t = 1
    while tile * t - (tile - 1) < window:
        t += 1
    return t


def _allowed(i: int, j: int, causal: bool, band=None) -> bool:
    if not causal:
        return True
    return j <= i and (band is None or i - j < band)


def visit_q(schedule: str, n: int, causal: bool, j: int, band=None) -> list:
    """Q tiles visited by KV tile j, in order (non-symmetric schedules).

    With a band (sliding window), tiles outside it are skipped as the
    masked tiles of a causal mask are; symmetric shift is then read as shift
    (all tasks but the last few have the same length, so there is no
    triangle to fold)."""
    if schedule in ("serialized_ascending", "atomic_nondet"):
        return [i for i in range(n) if _allowed(i, j, causal, band)]
    if schedule == "descending_q":
        return [i for i in reversed(range(n)) if _allowed(i, j, causal, band)]
    if schedule == "shift" or (schedule == "symmetric_shift" and (not causal or band is not None)):
        rot = [(j + t) % n for t in range(n)]
        return [i for i in rot if _allowed(i, j, causal, band)]
    raise ValueError(schedule)


def symmetric_task(n: int, jp: int):
    """Visit list of symmetric-shift task jp as (kv, q) pairs for ONE head.

    Returns (part_a, part_b): part_a is KV jp's phase 1 + phase 2a, part_b
    is KV n-1-jp's phase 2b (empty for the middle task of an odd n).
    """
    h = n // 2
    if n % 2 == 1 and jp == h:                      # middle tile, own task
        return [(jp, i) for i in range(n - 1, jp - 1, -1)], []
    a = [(jp, (n - h) + ((jp + t) % h)) for t in range(h)]        # phase 1
    a += [(jp, i) for i in range(jp, n - h)]                       # phase 2a
    m = n - 1 - jp
    b = [(m, i) for i in range(n - 1, m - 1, -1)]                  # phase 2b
    return a, b


def make_tasks(schedule: str, B: int, Hq: int, Hkv: int, n: int, causal: bool, band=None, nkv=None) -> list:
    """All tasks in dispatch order; each task is a list of Pair in run order."""
    if schedule not in SCHEDULES:
        raise ValueError(schedule)
    G = Hq // Hkv
    tasks = []
    for b in range(B):
        for hk in range(Hkv):
            heads = range(hk * G, (hk + 1) * G)
            if schedule == "symmetric_shift" and causal and band is None:
                for jp in range((n + 1) // 2):
                    a, bb = symmetric_task(n, jp)
                    t = [Pair(b, hq, i, kv) for hq in heads for (kv, i) in a]
                    t += [Pair(b, hq, i, kv) for hq in heads for (kv, i) in bb]
                    tasks.append(t)
            else:
                for j in range(n if nkv is None else nkv):
                    tasks.append([Pair(b, hq, i, j) for hq in heads
                                  for i in visit_q(schedule, n, causal, j, band)])
    # a band that reaches every tile of the causal triangle visits what the
    # causal mask visits, and is dealt like it
    banded = band is not None and band < n
    if schedule == "shift" and causal and not banded:
        # causal shift is dealt KV-tile-major: task k is KV tile k // (B*Hkv) of
        # head group k % (B*Hkv), so that each wave holds tiles of similar length
        groups = B * Hkv
        tasks = [tasks[g * n + j] for j in range(n) for g in range(groups)]
    elif schedule in STATIC and nkv is None and (banded or not causal or schedule == "symmetric_shift"):
        # shift on a full mask or a band, and symmetric shift (full or causal),
        # are dealt by the parity of the task's tile (pair) index: the even
        # tiles of every head group first, then the odd ones.  Within a wave a
        # dQ tile then receives a contribution every second step of the
        # rotation instead of every step, while the task -> worker rule stays
        # k -> k mod P.
        groups = B * Hkv
        T = len(tasks) // groups
        tasks = [tasks[g * T + t] for par in range(2) for g in range(groups) for t in range(par, T, 2)]
    return tasks


def build(schedule: str, B: int, Hq: int, Hkv: int, n: int, causal: bool, P: int, band=None,
          nkv=None) -> Schedule:
    """Tasks, assignment and accumulation order of a schedule (band: tile
    diagonals of a sliding window, from band_tiles, or None; nkv: key/value
    tiles per head when the key length differs from the query length, full
    masks only -- one task per KV tile, visiting all n query tiles, shift
    rotating from query tile kv mod n)."""
    if band is not None and (not causal or band < 1):
        raise ValueError("a band needs a causal mask and band >= 1")
    if nkv is not None and (causal or nkv < 1):
        raise ValueError("S_q != S_kv needs a full mask")
    tasks = make_tasks(schedule, B, Hq, Hkv, n, causal, band, nkv)
    static = schedule in STATIC
    s = Schedule(schedule, B, Hq, Hkv, n, causal, P, tasks, static)
    if static:
        s.cta_tasks = [list(range(c, len(tasks), P)) for c in range(P)]
        key = {}
        for c in range(P):
            t = 0
            for k in s.cta_tasks[c]:
                for p in tasks[k]:
                    key[p] = (t, p.j)      # model time, then lower KV index
                    t += 1
        per_tile = defaultdict(list)
        for p in key:
            per_tile[(p.b, p.hq, p.i)].append(p)
        s.turn = {tile: [p.j for p in sorted(ps, key=key.__getitem__)]
                  for tile, ps in per_tile.items()}
    elif schedule != "atomic_nondet":
        per_tile = defaultdict(list)
        for t in tasks:
            for p in t:
                per_tile[(p.b, p.hq, p.i)].append(p.j)
        s.turn = {tile: sorted(js) for tile, js in per_tile.items()}
    return s


def turn_ranks(s: Schedule) -> dict:
    """Pair -> rank of its reduction in its dQ tile's accumulation order."""
    out = {}
    if s.turn is None:
        return out
    for (b, hq, i), js in s.turn.items():
        for r, j in enumerate(js):
            out[Pair(b, hq, i, j)] = r
    return out


# --------------------------------------------------------------------------
# simulation with costs c (compute) and r (reduce)
# --------------------------------------------------------------------------

def simulate(s: Schedule, c: float, r: float) -> SimResult:
    """Event times of the DAG; raises RuntimeError on a deadlock."""
    ranks = turn_ranks(s)
    order = s.turn
    reduce_end: dict = {}
    if s.static:
        seqs = [[p for k in s.cta_tasks[cta] for p in s.tasks[k]] for cta in range(s.P)]
        cta_of_task = [k % s.P for k in range(len(s.tasks))]
        reduce_end = _longest_static(seqs, ranks, order, c, r)
    else:
        free = [0.0] * s.P
        cta_of_task = []
        for task in s.tasks:
            cta = min(range(s.P), key=lambda x: (free[x], x))
            cta_of_task.append(cta)
            t = free[cta]
            for p in task:
                ce = t + c
                rs = ce
                if order is not None and ranks[p] > 0:
                    pred = Pair(p.b, p.hq, p.i, order[(p.b, p.hq, p.i)][ranks[p] - 1])
                    if pred not in reduce_end:
                        raise RuntimeError("predecessor not yet dispatched: %r" % (pred,))
                    rs = max(rs, reduce_end[pred])
                t = rs + r
                reduce_end[p] = t
            free[cta] = t
    makespan = max(reduce_end.values()) if reduce_end else 0.0
    arrival = defaultdict(list)
    for p, t in reduce_end.items():
        arrival[(p.b, p.hq, p.i)].append((t, p.j))
    arrival = {tile: [j for _, j in sorted(v)] for tile, v in arrival.items()}
    return SimResult(makespan, cta_of_task, reduce_end, arrival)


def _longest_static(seqs, ranks, order, c, r):
    """Longest path over the chain + accumulation-order DAG (Kahn's algorithm).

    Node = pair (its reduce start is computed).  Edges: previous pair on the
    same SM (its reduce end -> this compute start) and the accumulation
    predecessor (its reduce end -> this reduce start).
    """
    prev_on_cta = {}
    for seq in seqs:
        for a, b in zip(seq, seq[1:]):
            prev_on_cta[b] = a
    preds = defaultdict(list)
    for p in ranks:
        k = ranks[p]
        if k > 0:
            tile = (p.b, p.hq, p.i)
            preds[p].append(("turn", Pair(p.b, p.hq, p.i, order[tile][k - 1])))
    for b, a in prev_on_cta.items():
        preds[b].append(("chain", a))
    nodes = [p for seq in seqs for p in seq]
    succ = defaultdict(list)
    indeg = {p: 0 for p in nodes}
    for p in nodes:
        for _, q in preds[p]:
            succ[q].append(p)
            indeg[p] += 1
    ready = deque(p for p in nodes if indeg[p] == 0)
    end = {}
    while ready:
        p = ready.popleft()
        cs = 0.0
        rs_floor = 0.0
        for kind, q in preds[p]:
            if kind == "chain":
                cs = max(cs, end[q])
            else:
                rs_floor = max(rs_floor, end[q])
        end[p] = max(cs + c, rs_floor) + r
        for q in succ[p]:
            indeg[q] -= 1
            if indeg[q] == 0:
                ready.append(q)
    if len(end) != len(nodes):
        raise RuntimeError("deadlock: the accumulation order and the SM chains form a cycle")
    return end


def check_tables(seqs, ranks) -> bool:
    """True if per-SM pair sequences + explicit ranks can all complete.

    ``seqs``: list (per SM) of lists of Pair; ``ranks``: Pair -> rank.  A dQ
    tile whose ranks are not exactly 0..m-1 has a missing predecessor; a
    cycle between chains and accumulation edges is a deadlock.  Either way
    the answer is False.
    """
    per_tile = defaultdict(list)
    for p, k in ranks.items():
        per_tile[(p.b, p.hq, p.i)].append((k, p.j))
    order = {}
    for tile, v in per_tile.items():
        v.sort()
        if [k for k, _ in v] != list(range(len(v))):
            return False
        order[tile] = [j for _, j in v]
    try:
        _longest_static(seqs, ranks, order, 1.0, 1.0)
    except RuntimeError:
        return False
    return True


# --------------------------------------------------------------------------
# the zero-weight-edge lemma (summary section 2.2.B)
# --------------------------------------------------------------------------

def depths(num_nodes: int, edges) -> list | None:
    """Longest-path depth of every node (sources at 0); None if cyclic.

    ``edges``: iterable of (u, v, w) meaning v starts at least w after u.
    """
    succ = defaultdict(list)
    indeg = [0] * num_nodes
    for u, v, w in edges:
        succ[u].append((v, w))
        indeg[v] += 1
    d = [0] * num_nodes
    ready = deque(x for x in range(num_nodes) if indeg[x] == 0)
    seen = 0
    while ready:
        u = ready.popleft()
        seen += 1
        for v, w in succ[u]:
            d[v] = max(d[v], d[u] + w)
            indeg[v] -= 1
            if indeg[v] == 0:
                ready.append(v)
    return d if seen == num_nodes else None


def critical_path(num_nodes: int, edges) -> int:
    d = depths(num_nodes, edges)
    if d is None:
        raise RuntimeError("cycle")
    return max(d) if d else 0


def add_zero_edge(num_nodes: int, edges, u: int, v: int):
    """Effect of adding the zero-weight edge u -> v.

    Returns (depths_unchanged, critical_path_unchanged) or None if the edge
    would close a cycle.
    """
    d0 = depths(num_nodes, edges)
    e1 = list(edges) + [(u, v, 0)]
    d1 = depths(num_nodes, e1)
    if d1 is None:
        return None
    return d0 == d1, max(d0) == max(d1)
