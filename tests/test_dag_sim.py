"""Pins for the schedule definitions and the DAG simulator (CPU only).

The closed forms are those printed in DASH overview (zskr.cn) section 3 for m
heads on n SMs; the cyclic order is the one printed in its section 3.2.
"""
import os

import pytest

from oracle import dag_sim as d

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

COSTS = [(3, 1), (1, 1), (5, 2), (7, 1), (4, 1)]


def makespan(mode, m, n, causal, P, c, r):
    return d.simulate(d.all_chains(mode, m, n, causal), P, c, r, ordered=(mode != "atomic")).makespan


@pytest.mark.parametrize("n", [4, 8, 16])
@pytest.mark.parametrize("m", [2, 4, 6])
@pytest.mark.parametrize("c,r", COSTS)
def test_closed_forms_at_P_equals_n(n, m, c, r):
    assert makespan("serial", m, n, True, n, c, r) == d.t_causal_serial(m, n, c, r)
    assert makespan("shift", m, n, False, n, c, r) == d.t_full_opt(m, n, c, r)
    assert makespan("symmetric_shift", m, n, True, n, c, r) == d.t_causal_opt(m, n, c, r)
    # written with "approximately" on the page; exact under the model when c >= r
    assert makespan("descending_q", m, n, True, n, c, r) == d.t_reversed(m, n, c, r)


@pytest.mark.parametrize("n,m,c,r", [(4, 4, 1, 3), (8, 2, 1, 2), (4, 2, 1, 5)])
def test_descending_formula_is_a_lower_bound_when_r_exceeds_c(n, m, c, r):
    assert makespan("descending_q", m, n, True, n, c, r) >= d.t_reversed(m, n, c, r)


def test_shift_order_matches_printed_cycle():
    rows = [list(map(int, ln.split())) for ln in open(os.path.join(GOLDEN, "shift_order_n4.txt"))
            if ln.strip() and not ln.startswith("#")]
    chains = d.head_chains("shift", 4, False)
    assert [[q for (kv, q) in ch] for ch in chains] == rows
    assert [[kv for (kv, q) in ch] for ch in chains] == [[i] * 4 for i in range(4)]


@pytest.mark.parametrize("n", [2, 4, 6, 8, 16, 32, 128])
def test_symmetric_shift_covers_causal_triangle_once(n):
    chains = d.head_chains("symmetric_shift", n, True)
    assert len(chains) == n // 2
    assert all(len(ch) == n + 1 for ch in chains)
    seen = [t for ch in chains for t in ch]
    assert sorted(seen) == sorted((kv, q) for kv in range(n) for q in range(kv, n))
    # phase 1 is the dense lower-left block: KV < n/2, Q >= n/2
    for p, ch in enumerate(chains):
        assert all(kv == p and q >= n // 2 for kv, q in ch[: n // 2])
        assert all(kv == n - 1 - p for kv, q in ch[n - p:])
    d.head_ranks("symmetric_shift", n, True)   # raises if two chains meet a tile at one step


@pytest.mark.parametrize("mode,causal", [("atomic", False), ("atomic", True), ("serial", False),
                                         ("serial", True), ("descending_q", False),
                                         ("descending_q", True), ("shift", False)])
@pytest.mark.parametrize("n", [1, 3, 8])
def test_chains_cover_mask_and_ranks_are_permutations(mode, causal, n):
    chains = d.head_chains(mode, n, causal)
    seen = sorted(t for ch in chains for t in ch)
    want = sorted((kv, q) for kv in range(n) for q in range(n) if (q >= kv or not causal))
    assert seen == want
    ranks = d.head_ranks(mode, n, causal, chains)
    per_q = {}
    for ch, rk in zip(chains, ranks):
        assert len({kv for kv, _ in ch}) == 1           # KV-stationary
        for (kv, q), r in zip(ch, rk):
            per_q.setdefault(q, []).append(r)
    for q, rs in per_q.items():
        assert sorted(rs) == list(range(len(rs)))
    if mode == "descending_q":
        assert all([q for _, q in ch] == sorted((q for _, q in ch), reverse=True) for ch in chains)


@pytest.mark.parametrize("mode,causal", [("shift", False), ("symmetric_shift", True)])
@pytest.mark.parametrize("n,m", [(4, 4), (8, 2), (16, 6)])
def test_lemma1_conflict_free_schedules_never_wait(mode, causal, n, m):
    # Lemma 1 (gist.science/it, section 2.2 B): ordering edges that go from a
    # node to one of no smaller depth keep the critical path.  The shift
    # schedules build such an order, so no R stage ever waits at P = n.
    sim = d.simulate(d.all_chains(mode, m, n, causal), n, 4, 1)
    assert all(sim.r_start[t] == sim.c_end[t] for t in sim.c_end)
    # and every ordered predecessor's R has ended when the successor's C ends
    chains = d.all_chains(mode, m, n, causal)
    by_tile = {}
    for ci, (bh, ch, rk) in enumerate(chains):
        for st, ((kv, q), rank) in enumerate(zip(ch, rk)):
            by_tile.setdefault((bh, q), {})[rank] = (ci, st)
    for tile, mm in by_tile.items():
        for rank in range(1, len(mm)):
            assert sim.r_end[mm[rank - 1]] <= sim.c_end[mm[rank]]


def test_serial_waits_exist():
    sim = d.simulate(d.all_chains("serial", 2, 8, True), 8, 4, 1)
    assert any(sim.r_start[t] > sim.c_end[t] for t in sim.c_end)


def test_shift_needs_a_whole_gang():
    with pytest.raises(d.Deadlock):
        d.simulate(d.all_chains("shift", 1, 8, False), 4, 4, 1)
    d.simulate(d.all_chains("serial", 1, 8, False), 4, 4, 1)       # serial does not


def test_invalid_modes_rejected():
    with pytest.raises(d.ScheduleError):
        d.head_chains("shift", 4, True)
    with pytest.raises(d.ScheduleError):
        d.head_chains("symmetric_shift", 4, False)
    with pytest.raises(d.ScheduleError):
        d.head_chains("symmetric_shift", 5, True)


def test_tables_flags_and_order():
    tasks, off, ms = d.schedule_tables("symmetric_shift", 3, 4, True, 5)
    assert off[0] == 0 and off[-1] == len(tasks) == 3 * 10
    # each chain of symmetric shift holds two KV runs: first/last flags bracket each
    for s in range(5):
        run = tasks[off[s]:off[s + 1]]
        for i, (bh, kv, q, w) in enumerate(run):
            first = i == 0 or run[i - 1][1] != kv or run[i - 1][0] != bh
            last = i == len(run) - 1 or run[i + 1][1] != kv or run[i + 1][0] != bh
            assert bool(w & d.FLAG_FIRST) == first
            assert bool(w & d.FLAG_LAST) == last


def head_rank_map(mode, n, causal):
    chains = d.head_chains(mode, n, causal)
    ranks = d.head_ranks(mode, n, causal, chains)
    return {t: rk for ch, rks in zip(chains, ranks) for t, rk in zip(ch, rks)}


@pytest.mark.parametrize("mode,causal,BH,n,P,c,r", [
    ("shift", False, 32, 32, 152, 4, 1), ("shift", False, 32, 32, 152, 1, 1), ("shift", False, 7, 4, 10, 4, 1),
    ("shift", False, 9, 6, 20, 2, 3), ("shift", False, 16, 8, 20, 1, 2), ("shift", False, 13, 5, 12, 3, 1),
    ("symmetric_shift", True, 16, 8, 10, 4, 1), ("symmetric_shift", True, 16, 8, 10, 1, 1),
    ("symmetric_shift", True, 11, 6, 14, 1, 3), ("symmetric_shift", True, 12, 16, 36, 2, 1)])
def test_fill_split(mode, causal, BH, n, P, c, r):
    # fill (an extension): every tile of every head once, each head with its
    # own schedule's ranks, CTAs within the budget, the leftover CTAs holding
    # only filled heads, and no split of the heads (whole waves or not) or
    # fill schedule with a smaller makespan
    tasks, off, ms, hs, fm = d.fill_tables(mode, BH, n, causal, P, c, r)
    tiles = [(kv, q) for kv in range(n) for q in range(n) if not causal or q >= kv]
    assert sorted((bh, kv, q) for bh, kv, q, _ in tasks) == [(bh, kv, q) for bh in range(BH) for kv, q in tiles]
    assert len(off) - 1 <= P and off[0] == 0 and off[-1] == len(tasks)
    assert all(a <= b for a, b in zip(off, off[1:]))
    own = head_rank_map(mode, n, causal)
    other = head_rank_map(fm, n, causal) if fm else None
    for bh, kv, q, w in tasks:
        assert (w & d.RANK_MASK) == (own if bh < hs else other)[(kv, q)]
    gang = n // 2 if mode == "symmetric_shift" else n
    per_wave, F = P // gang, P % gang
    assert per_wave and F and BH > per_wave, "the case must exercise the fill"
    fills = ("serial", "descending_q") if causal else ("serial",)
    brute = min(max(makespan(mode, h, n, causal, min(per_wave * gang, h * gang), c, r),
                    min(makespan(f, BH - h, n, causal, min(F, (BH - h) * n), c, r) for f in fills) if h < BH else 0)
                for h in range(1, BH + 1))
    assert ms == brute
    first_fill_cta = min(per_wave * gang, hs * gang)
    assert all(tasks[i][0] >= hs for i in range(off[first_fill_cta], len(tasks)))


def test_fill_is_plain_shift_without_leftover_ctas():
    tasks, off, ms, hs, fm = d.fill_tables("shift", 8, 4, False, 16, 4, 1)   # 16 = 4 whole gangs
    assert (hs, fm) == (8, None)
    assert (tasks, off, ms) == d.schedule_tables("shift", 8, 4, False, 16, 4, 1)


# ---- split gangs (an extension beyond the pages' schedules)

@pytest.mark.parametrize("mode,causal,n", [("shift", False, 8), ("shift", False, 12), ("symmetric_shift", True, 8),
                                           ("symmetric_shift", True, 16)])
@pytest.mark.parametrize("split", [1, 2, 4])
def test_split_gangs_cover_the_mask_and_order_tiles_by_subgang(mode, causal, n, split):
    BH = 3
    gang = n if mode == "shift" else n // 2
    if gang % split:
        with pytest.raises(d.ScheduleError):
            d.split_chains(mode, BH, n, causal, split)
        return
    chains = d.split_chains(mode, BH, n, causal, split)
    g = gang // split
    # dispatch order: sub-gang 0 of every head, then sub-gang 1, ...
    heads = [bh for bh, _, _ in chains]
    assert heads == [bh for _ in range(split) for bh in range(BH) for _ in range(g)]
    # the same tasks as the whole gangs: every (head, kv, q) of the mask once
    plain = {(bh, kv, q) for bh, ch, _ in d.all_chains(mode, BH, n, causal) for kv, q in ch}
    got = [(bh, kv, q) for bh, ch, _ in chains for kv, q in ch]
    assert len(got) == len(set(got)) and set(got) == plain
    # per tile the ranks are 0..k-1, and a sub-gang's ranks follow all of the one before it
    by_tile = {}
    for i, (bh, ch, rk) in enumerate(chains):
        for (kv, q), rank in zip(ch, rk):
            by_tile.setdefault((bh, q), []).append((rank, i // (BH * g)))
    for tile, lst in by_tile.items():
        ranks = sorted(r for r, _ in lst)
        assert ranks == list(range(len(lst)))
        subs_in_rank_order = [s for _, s in sorted(lst)]
        assert subs_in_rank_order == sorted(subs_in_rank_order)
    if split == 1:   # no split: exactly the pages' order
        assert [rk for _, _, rk in chains] == [rk for _, _, rk in d.all_chains(mode, BH, n, causal)]


@pytest.mark.parametrize("mode,causal,n,m", [("shift", False, 8, 3), ("shift", False, 16, 2),
                                             ("symmetric_shift", True, 8, 3), ("symmetric_shift", True, 16, 2)])
@pytest.mark.parametrize("split", [2, 4])
@pytest.mark.parametrize("c,r", [(4, 1), (3, 2), (1, 1)])
def test_split_gangs_never_wait_on_one_subgang_of_sms(mode, causal, n, m, split, c, r):
    # with as many SMs as a sub-gang, sub-gangs run one after another in
    # lockstep: no R waits, so the makespan is m * split sub-gangs of one
    # chain length each, (c + r) per task (n tasks for shift, n + 1 for
    # symmetric shift: the closed forms' T_full_opt and T_causal_opt per gang)
    gang = n if mode == "shift" else n // 2
    g = gang // split
    sim = d.simulate(d.split_chains(mode, m, n, causal, split), g, c, r)
    length = n if mode == "shift" else n + 1
    assert sim.makespan == m * split * length * (c + r)
    assert all(sim.r_start[t] == sim.c_end[t] for t in sim.c_end)


def test_split_tables_of_one_equal_the_plain_tables():
    for mode, causal, n, P in (("shift", False, 8, 16), ("symmetric_shift", True, 8, 12)):
        a = d.split_tables(mode, 3, n, causal, 1, P, 4, 1)
        b = d.schedule_tables(mode, 3, n, causal, P, 4, 1)
        assert a == b


# ---- timed ranks (an extension beyond the pages' orders)

@pytest.mark.parametrize("mode,causal,n,BH,P", [("shift", False, 8, 4, 8), ("shift", False, 8, 4, 16),
                                                ("shift", False, 8, 4, 32), ("shift", False, 6, 3, 12),
                                                ("symmetric_shift", True, 8, 4, 4), ("symmetric_shift", True, 8, 4, 12),
                                                ("symmetric_shift", True, 16, 3, 16)])
def test_timed_ranks_are_the_pages_ranks_for_whole_gangs_side_by_side(mode, causal, n, BH, P):
    # whole gangs side by side (P a multiple of the gang) run in lockstep, so
    # the order in which they reach a tile is its visiting-step order: the
    # pages' ranks, bit for bit, and the same tables
    chains = d.all_chains(mode, BH, n, causal)
    timed = d.timed_chains(chains, P, 4, 1)
    assert [rk for _, _, rk in timed] == [rk for _, _, rk in chains]
    assert d.timed_tables(mode, BH, n, causal, P) == d.schedule_tables(mode, BH, n, causal, P)


@pytest.mark.parametrize("mode,causal,n,BH,P,split", [("shift", False, 8, 5, 12, 1), ("shift", False, 8, 5, 12, 2),
                                                      ("symmetric_shift", True, 16, 3, 10, 1),
                                                      ("symmetric_shift", True, 16, 5, 12, 2),
                                                      ("serial", False, 6, 4, 7, 1), ("descending_q", True, 8, 3, 9, 1)])
@pytest.mark.parametrize("c,r", [(4, 1), (1, 3)])
def test_timed_ranks_permute_each_tile_and_follow_the_schedule(mode, causal, n, BH, P, split, c, r):
    base = d.split_chains(mode, BH, n, causal, split) if split > 1 else d.all_chains(mode, BH, n, causal)
    timed = d.timed_chains(base, P, c, r)
    # same chains and tasks, new ranks: each (head, q) tile's ranks are 0..k-1
    assert [(bh, ch) for bh, ch, _ in timed] == [(bh, ch) for bh, ch, _ in base]
    by_tile = {}
    for bh, ch, rk in timed:
        for (kv, q), x in zip(ch, rk):
            by_tile.setdefault((bh, q), []).append(x)
    assert all(sorted(v) == list(range(len(v))) for v in by_tile.values())
    # the ranks follow the unordered run's compute ends, and the ordered run of
    # the timed ranks completes (a deadlock raises) no later than the
    # unordered run plus one reduction per task of the longest chain
    free = d.simulate(base, P, c, r, ordered=False)
    for ci, (bh, ch, rk) in enumerate(timed):
        for st, ((kv, q), x) in enumerate(zip(ch, rk)):
            for cj, (bh2, ch2, rk2) in enumerate(timed):
                if bh2 != bh:
                    continue
                for st2, ((kv2, q2), x2) in enumerate(zip(ch2, rk2)):
                    if q2 == q and x2 < x:
                        assert (free.c_end[(cj, st2)], cj, st2) < (free.c_end[(ci, st)], ci, st)
    ordered = d.simulate(timed, P, c, r)
    longest = max(len(ch) for _, ch, _ in base)
    assert ordered.makespan <= free.makespan + longest * r * BH


@pytest.mark.parametrize("mode,causal", [("serial", False), ("descending_q", False), ("descending_q", True)])
@pytest.mark.parametrize("n,BH", [(4, 2), (8, 3)])
def test_timed_ranks_of_serial_and_descending_with_every_chain_at_once(mode, causal, n, BH):
    # with a CTA per chain every chain starts at time 0; in these schedules all the chains of a head reach a tile
    # at the same step, so the tie goes to the dispatch position, ascending KV: the pages' order
    chains = d.all_chains(mode, BH, n, causal)
    timed = d.timed_chains(chains, len(chains), 4, 1)
    assert [rk for _, _, rk in timed] == [rk for _, _, rk in chains]


@pytest.mark.parametrize("n,BH", [(4, 2), (8, 3)])
def test_timed_ranks_of_causal_serial_run_in_descending_kv(n, BH):
    # causal serial: KV j starts at tile j, so with a CTA per chain KV q reaches tile q first and KV 0 last; the
    # timed order is descending KV, where the pages' order (ascending KV) makes every chain wait on KV 0's
    chains = d.all_chains("serial", BH, n, True)
    timed = d.timed_chains(chains, len(chains), 4, 1)
    for bh, ch, rk in timed:
        for (kv, q), x in zip(ch, rk):
            assert x == q - kv
