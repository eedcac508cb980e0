"""DASH schedules and the DAG critical-path simulator, written from the pages.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark import
this module.  The CUDA library's host schedule generator is a separate C++
implementation of the same definitions; the tests compare the two tables
element by element.

Model (DASH overview (zskr.cn), section 2.2; Sintesi Tecnica DASH
(gist.science/it), section 2.1).  The backward is a DAG whose nodes are compute
stages C (one KV tile against one Q tile, cost c) and reduction stages R (adding
that task's dQ partial into the dQ tile, cost r).  All work on one KV tile runs
back to back on one SM ("unbroken chains"), so a chain is the list of Q tiles one
KV tile visits, and each task of a chain is C followed by R.  Determinism fixes,
for every dQ tile, the order in which the R stages that touch it run: R of a
task waits until the R of its predecessor in that order has finished.  The goal
is the shortest critical path.

Readings taken where the pages are silent (each is also listed in the design
notes):
  * n is at once the number of KV blocks, of Q tiles and, in the closed forms,
    of SMs (overview, section 3.1: "m heads, n SMs").
  * Chains are dispatched in (head, slot) order; each goes to the SM that falls
    idle first, ties to the lowest SM id; a chain occupies its SM until its
    last R ends (waits included).
  * Serial and descending reduce each dQ tile in ascending KV order (the
    FlashAttention-3 "relay baton" order, overview section 2.1).
  * Shift: chain j (KV tile j) visits Q tiles (j + t) mod n for t = 0..n-1, the
    cyclic order of overview section 3.2 read as KV-stationary; a dQ tile is
    reduced in visiting-step order.
  * Symmetric shift (overview section 3.3; gist.science/it section 2.2B): slot
    p < n/2 owns KV p and KV n-1-p.  Phase 1 (dense lower-left rectangle):
    KV p, Q tiles n/2 + ((p + t) mod n/2), t < n/2.  Phase 2 (the folded
    triangle): KV p, Q tiles p .. n/2-1 ascending; then KV n-1-p, Q tiles
    n-1 down to n-1-p.  A dQ tile is reduced in visiting-step order.
  * Atomic: the serial chains with no ordering between R stages.

Pins (tests/test_dag_sim.py): the four closed forms of overview section 3
at P = n, the cyclic visiting order printed in overview section 3.2
(tests/golden/shift_order_n4.txt), Lemma 1's consequence that the
conflict-free schedules never wait at P = n, and coverage of every tile.
fill_tables (an extension) is pinned by coverage, by each head's ranks
equalling its own schedule's, and by brute force over every split of the
heads; fit_costs by recovering the r that produced simulated makespans.
split_chains (an extension) is pinned by coverage, by each tile's ranks
running sub-gang after sub-gang, by equality with the plain chains for a split
of one, and by the closed form m * split * len * (c + r) with no wait on as
many SMs as a sub-gang (the overview's optimal forms, section 3, per gang).
timed_chains (an extension) is pinned by equality with the pages' ranks where
whole shift gangs run side by side (the step order is then the time order), by
ranks that are permutations of every tile's visits, and by a run that never
waits longer than its own reduction order allows.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass

MODES = ("atomic", "serial", "descending_q", "shift", "symmetric_shift")
MODE_ID = {m: i for i, m in enumerate(MODES)}

FLAG_FIRST = 1 << 28   # first task of a run on one KV tile: accumulators start at zero
FLAG_LAST = 1 << 29    # last task of a run on one KV tile: dK/dV are written out
RANK_MASK = (1 << 24) - 1


class ScheduleError(ValueError):
    pass


class Deadlock(RuntimeError):
    pass


def check_mode(mode: str, n: int, causal: bool):
    if mode not in MODES:
        raise ScheduleError(f"unknown schedule {mode!r}")
    if n < 1:
        raise ScheduleError("n must be >= 1")
    if mode == "shift" and causal:
        raise ScheduleError("shift scheduling is defined for full masks only")
    if mode == "symmetric_shift":
        if not causal:
            raise ScheduleError("symmetric shift is defined for causal masks only")
        if n % 2:
            raise ScheduleError("symmetric shift pairs KV i with n-1-i: n must be even")


def head_chains(mode: str, n: int, causal: bool):
    """The chains of one head, in slot order.  Each chain is a list of
    (kv, q) block pairs in visiting order."""
    check_mode(mode, n, causal)
    chains = []
    if mode in ("atomic", "serial"):
        for j in range(n):
            first_q = j if causal else 0
            chains.append([(j, q) for q in range(first_q, n)])
    elif mode == "descending_q":
        for j in range(n):
            last_q = j if causal else 0
            chains.append([(j, q) for q in range(n - 1, last_q - 1, -1)])
    elif mode == "shift":
        for j in range(n):
            chains.append([(j, (j + t) % n) for t in range(n)])
    else:  # symmetric_shift
        h = n // 2
        for p in range(h):
            ch = [(p, h + (p + t) % h) for t in range(h)]          # phase 1
            ch += [(p, q) for q in range(p, h)]                      # phase 2, KV p
            ch += [(n - 1 - p, n - 1 - i) for i in range(p + 1)]     # phase 2, KV n-1-p
            chains.append(ch)
    return chains


def head_ranks(mode: str, n: int, causal: bool, chains=None):
    """Rank of every task of one head in its dQ tile's reduction order, as a
    list of lists parallel to ``head_chains``."""
    if chains is None:
        chains = head_chains(mode, n, causal)
    if mode in ("atomic", "serial", "descending_q"):
        # ascending KV index; for causal only kv <= q visit q, so rank = kv
        return [[kv for (kv, q) in ch] for ch in chains]
    # shift / symmetric shift: order of the visiting step, conflict-free
    visits = {}
    for slot, ch in enumerate(chains):
        for step, (kv, q) in enumerate(ch):
            visits.setdefault(q, []).append((step, slot))
    rank_of = {}
    for q, lst in visits.items():
        steps = [s for s, _ in lst]
        if len(set(steps)) != len(steps):
            raise ScheduleError(f"two chains reach dQ tile {q} at the same step")
        for rk, (step, slot) in enumerate(sorted(lst)):
            rank_of[(slot, step)] = rk
    return [[rank_of[(slot, step)] for step in range(len(ch))] for slot, ch in enumerate(chains)]


@dataclass
class Simulation:
    makespan: int
    sm_of_chain: list        # chain index -> SM
    chains_of_sm: list       # SM -> chain indices in run order
    chain_start: list
    chain_finish: list
    c_end: dict              # (chain, step) -> time C ends
    r_start: dict            # (chain, step) -> time R starts
    r_end: dict              # (chain, step) -> time R ends


def all_chains(mode: str, BH: int, n: int, causal: bool):
    """Chains of every head in dispatch order (head-major, then slot), with
    their head index and ranks: a list of (bh, [(kv, q)], [rank])."""
    hc = head_chains(mode, n, causal)
    hr = head_ranks(mode, n, causal, hc)
    return [(bh, hc[s], hr[s]) for bh in range(BH) for s in range(len(hc))]


def simulate(chains, P: int, c: int, r: int, ordered: bool = True) -> Simulation:
    """Discrete-event list scheduling of the chains on P SMs.

    ``chains`` is the output of ``all_chains``.  Integer costs c, r >= 1.  At
    time 0 SMs 0..P-1 take the first chains in order; afterwards an SM that
    falls idle at time T takes the next chain at T (ties: lowest SM id first).
    A task's R starts when its C has ended and, if ``ordered``, when the R of
    its predecessor in the dQ tile's order has ended.  Raises Deadlock when no
    SM can make progress.
    """
    if c < 1 or r < 1 or P < 1:
        raise ValueError("costs and P must be >= 1")
    pred = {}
    if ordered:
        by_tile = {}
        for ci, (bh, ch, rk) in enumerate(chains):
            for st, ((kv, q), rank) in enumerate(zip(ch, rk)):
                by_tile.setdefault((bh, q), {})[rank] = (ci, st)
        for tile, m in by_tile.items():
            for rank in range(1, len(m)):
                pred[m[rank]] = m[rank - 1]

    nch = len(chains)
    heap = []
    sm_chain = [-1] * P
    sm_step = [0] * P
    sm_phase = [""] * P
    sm_of_chain = [-1] * nch
    chains_of_sm = [[] for _ in range(P)]
    chain_start = [0] * nch
    chain_finish = [0] * nch
    c_end, r_start, r_end = {}, {}, {}
    waiting = {}
    nxt = 0

    def dispatch(s, t):
        nonlocal nxt
        ci = nxt
        nxt += 1
        sm_chain[s], sm_step[s], sm_phase[s] = ci, 0, "C"
        sm_of_chain[ci] = s
        chains_of_sm[s].append(ci)
        chain_start[ci] = t
        heapq.heappush(heap, (t + c, s))

    for s in range(P):
        if nxt < nch:
            dispatch(s, 0)
    makespan = 0
    while heap:
        T = heap[0][0]
        batch = []
        while heap and heap[0][0] == T:
            batch.append(heapq.heappop(heap)[1])
        freed = []
        for s in sorted(batch):
            task = (sm_chain[s], sm_step[s])
            if sm_phase[s] == "C":
                c_end[task] = T
                p = pred.get(task)
                if p is None or p in r_end:
                    sm_phase[s] = "R"
                    r_start[task] = T
                    heapq.heappush(heap, (T + r, s))
                else:
                    sm_phase[s] = "W"
                    waiting[p] = s
            else:
                r_end[task] = T
                w = waiting.pop(task, None)
                if w is not None:
                    sm_phase[w] = "R"
                    r_start[(sm_chain[w], sm_step[w])] = T
                    heapq.heappush(heap, (T + r, w))
                ci, st = task
                if st + 1 < len(chains[ci][1]):
                    sm_step[s] = st + 1
                    sm_phase[s] = "C"
                    heapq.heappush(heap, (T + c, s))
                else:
                    chain_finish[ci] = T
                    makespan = max(makespan, T)
                    sm_chain[s] = -1
                    sm_phase[s] = ""
                    freed.append(s)
        for s in sorted(freed):
            if nxt < nch:
                dispatch(s, T)
    if nxt < nch or waiting:
        raise Deadlock(f"{len(waiting)} SMs wait forever, {nch - nxt} chains never start")
    return Simulation(makespan, sm_of_chain, chains_of_sm, chain_start, chain_finish,
                      c_end, r_start, r_end)


def schedule_tables(mode: str, BH: int, n: int, causal: bool, P: int, c: int = 4, r: int = 1):
    """Per-CTA task tables for the GPU kernel, from the simulation on P SMs.

    Returns (tasks, cta_off, makespan): ``tasks`` is a flat list of int32
    quadruples (bh, kv, q, rank | flags) grouped by CTA, CTA s owning entries
    cta_off[s] .. cta_off[s+1]-1, in the order the simulation ran them.
    FLAG_FIRST marks the first task of a run on one KV tile, FLAG_LAST the
    last one.
    """
    return tables_of(all_chains(mode, BH, n, causal), P, c, r, ordered=(mode != "atomic"))


def split_chains(mode: str, BH: int, n: int, causal: bool, split: int):
    """Split gangs (an extension beyond the pages' schedules) of shift or
    symmetric shift.  Each head's gang of chains (slot order) runs as ``split``
    sub-gangs of consecutive slots.  The chains are dispatched sub-gang by
    sub-gang: sub-gang 0 of every head, then sub-gang 1 of every head, and so
    on.  A dQ tile's ranks go in (sub-gang, visiting step) order, so a
    sub-gang adds to a tile only after the sub-gangs before it are done with
    it; inside a sub-gang no two chains reach one tile at one step.  Returns
    the chains in dispatch order, as ``all_chains`` does."""
    if mode not in ("shift", "symmetric_shift"):
        raise ScheduleError("split gangs apply to shift and symmetric shift only")
    hc = head_chains(mode, n, causal)
    if split < 1 or len(hc) % split:
        raise ScheduleError("the split must divide the chains of a head's gang")
    g = len(hc) // split
    visits = {}
    for slot, ch in enumerate(hc):
        for step, (kv, q) in enumerate(ch):
            visits.setdefault(q, []).append((slot // g, step, slot))
    rank_of = {}
    for q, lst in visits.items():
        keys = [(sub, step) for sub, step, _ in lst]
        if len(set(keys)) != len(keys):
            raise ScheduleError(f"two chains of one sub-gang reach dQ tile {q} at the same step")
        for rk, (sub, step, slot) in enumerate(sorted(lst)):
            rank_of[(slot, step)] = rk
    hr = [[rank_of[(slot, step)] for step in range(len(ch))] for slot, ch in enumerate(hc)]
    return [(bh, hc[slot], hr[slot]) for sub in range(split) for bh in range(BH)
            for slot in range(sub * g, (sub + 1) * g)]


def split_tables(mode: str, BH: int, n: int, causal: bool, split: int, P: int, c: int = 4, r: int = 1):
    """``schedule_tables`` for split gangs (``split_chains``)."""
    return tables_of(split_chains(mode, BH, n, causal, split), P, c, r, ordered=True)


def timed_chains(chains, P: int, c: int, r: int):
    """Timed ranks (an extension beyond the pages' orders): every dQ tile is
    reduced in the order in which the scheduled chains reach it.  The chains
    (in dispatch order) are list-scheduled on P SMs without reduction order;
    the visits of each (head, q) tile are ranked by the time their compute
    stage ends, ties by the chain's dispatch position, then by step.  Returns
    the chains with those ranks."""
    sim = simulate(chains, P, c, r, ordered=False)
    visits = {}
    for ci, (bh, ch, _) in enumerate(chains):
        for st, (kv, q) in enumerate(ch):
            visits.setdefault((bh, q), []).append((sim.c_end[(ci, st)], ci, st))
    rank = {}
    for lst in visits.values():
        for rk, (_, ci, st) in enumerate(sorted(lst)):
            rank[(ci, st)] = rk
    return [(bh, ch, [rank[(ci, st)] for st in range(len(ch))]) for ci, (bh, ch, _) in enumerate(chains)]


def timed_tables(mode: str, BH: int, n: int, causal: bool, P: int, split: int = 1, c: int = 4, r: int = 1):
    """``schedule_tables`` with timed ranks (``timed_chains``), of whole gangs
    or of split gangs (``split_chains``)."""
    chains = split_chains(mode, BH, n, causal, split) if split > 1 else all_chains(mode, BH, n, causal)
    return tables_of(timed_chains(chains, P, c, r), P, c, r, ordered=True)


def tables_of(chains, P: int, c: int, r: int, ordered: bool):
    """Task tables of chains given in dispatch order (see ``schedule_tables``)."""
    sim = simulate(chains, P, c, r, ordered=ordered)
    tasks = []
    cta_off = [0]
    for s in range(P):
        for ci in sim.chains_of_sm[s]:
            bh, ch, rk = chains[ci]
            for st, ((kv, q), rank) in enumerate(zip(ch, rk)):
                w = rank
                if st == 0 or ch[st - 1][0] != kv:
                    w |= FLAG_FIRST
                if st == len(ch) - 1 or ch[st + 1][0] != kv:
                    w |= FLAG_LAST
                tasks.append((bh, kv, q, w))
        cta_off.append(len(tasks))
    return tasks, cta_off, sim.makespan


def fill_tables(mode: str, BH: int, n: int, causal: bool, P_max: int, c: int = 4, r: int = 1):
    """Fill: an extension beyond the pages' schedules, for shift (full mask) and
    symmetric shift (causal).

    A head's chains each wait on a neighbour in the head's gang (n chains for
    shift, n/2 for symmetric shift), so these schedules want whole gangs of
    SMs, and on P_max SMs that are not a multiple of the gang the rest idle.
    Here the heads split in two: the first hs heads run `mode` on
    G = (P_max // gang) * gang SMs, the others run a fill schedule on the
    P_max - G SMs left over (serial; for a causal mask serial or
    descending_q), each head keeping its own schedule's reduction order.
    hs ranges over whole waves of gangs (k * (P_max // gang), and BH); the
    split and fill schedule whose larger makespan is smallest win, ties to
    more shift heads, then to serial.  Without SMs left over, or when every
    head fits in one wave, this is plain `mode` on the CTA count that the
    library's CTA choice takes (for shift the smallest whole number of gangs
    with the best makespan; for symmetric shift also P_max itself).

    Returns (tasks, cta_off, makespan, shift_heads, fill_mode or None) like
    schedule_tables; the filled heads are numbered after the others and
    their CTAs come after theirs.
    """
    check_mode(mode, n, causal)
    if mode not in ("shift", "symmetric_shift"):
        raise ScheduleError("fill applies to shift and symmetric shift only")
    gang = n // 2 if mode == "symmetric_shift" else n
    per_wave = P_max // gang
    G = per_wave * gang
    F = P_max - G
    if per_wave == 0 or F == 0 or BH <= per_wave:
        top = min(P_max, BH * gang)
        cands = list(range((top // gang) * gang, gang - 1, -gang))
        if mode == "symmetric_shift":   # the CTA choice also offers the full count
            cands = [top] + [m for m in cands if m != top][:15]
        best = None
        for m in cands[:16]:
            try:
                ms = simulate(all_chains(mode, BH, n, causal), m, c, r).makespan
            except Deadlock:
                continue
            if best is None or ms < best[0] or (ms == best[0] and m < best[1]):
                best = (ms, m)
        if best is None:
            raise Deadlock("no CTA count runs this schedule without deadlock")
        tasks, off, ms = schedule_tables(mode, BH, n, causal, best[1], c, r)
        return tasks, off, ms, BH, None
    fills = ("serial", "descending_q") if causal else ("serial",)
    best = None
    for k in range(-(-BH // per_wave), 0, -1):
        hs = min(BH, k * per_wave)
        rest = BH - hs
        P1 = min(G, hs * gang)
        try:
            ms1 = simulate(all_chains(mode, hs, n, causal), P1, c, r).makespan
        except Deadlock:
            continue
        for fm in (fills if rest else (None,)):
            ms, P2 = ms1, 0
            if rest:
                P2 = min(F, rest * n)
                try:
                    ms = max(ms, simulate(all_chains(fm, rest, n, causal), P2, c, r).makespan)
                except Deadlock:
                    continue
            if best is None or ms < best[0]:
                best = (ms, hs, P1, P2, fm)
    if best is None:
        raise Deadlock("no split runs without deadlock")
    ms, hs, P1, P2, fm = best
    tasks, off, _ = schedule_tables(mode, hs, n, causal, P1, c, r)
    if P2:
        t2, off2, _ = schedule_tables(fm, BH - hs, n, causal, P2, c, r)
        tasks = tasks + [(bh + hs, kv, q, w) for (bh, kv, q, w) in t2]
        off = off + [off[-1] + x for x in off2[1:]]
    return tasks, off, ms, hs, fm


FIT_COST_C = 8
FIT_COST_R = (1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128, 192, 256, 384, 512)


def fit_costs(BH: int, n: int, causal: bool, P_max: int, atomic_ms: float, serial_ms: float):
    """Task costs from measured times: c = FIT_COST_C and the r of FIT_COST_R
    whose simulated serial / atomic makespan ratio (both on min(P_max, chains)
    SMs) is nearest serial_ms / atomic_ms, ties to the smaller r."""
    P = min(P_max, BH * n)
    want = serial_ms / atomic_ms
    best = None
    for r in FIT_COST_R:
        a = simulate(all_chains("atomic", BH, n, causal), P, FIT_COST_C, r, ordered=False).makespan
        s = simulate(all_chains("serial", BH, n, causal), P, FIT_COST_C, r).makespan
        err = abs(s / a - want)
        if best is None or err < best[0]:
            best = (err, r)
    return FIT_COST_C, best[1]


# Closed forms of DASH overview (zskr.cn) section 3, for m heads on n SMs.
def t_causal_serial(m, n, c, r):
    return m * n * (c + r) + (n - 1) * r


def t_reversed(m, n, c, r):
    """Written with "approximately" on the page; exact when c >= r under the
    model above."""
    return m * (n + 1) * (c + r) // 2 + (n - 1) * r


def t_full_opt(m, n, c, r):
    return m * n * (c + r)


def t_causal_opt(m, n, c, r):
    return m * (n + 1) * (c + r) // 2
