"""C-ABI checks that need no GPU: the library loads, exports every function
that include/dash.h declares, and its host schedule generator reproduces the
oracle simulator's tables element by element."""
import os
import re

import numpy as np
import pytest

import deterministic_attention_backward_fa_gb300 as dash
from oracle import dag_sim as d

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dash.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dash_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert "dash_attn_bwd" in names and "dash_attn_fwd" in names
    L = dash.lib()
    for n in names:
        assert hasattr(L, n), n
        assert n in dash.__dict__, f"binding lacks {n}"


CASES = [(m, c, n, BH, P) for m in d.MODES for c in (False, True) for n in (1, 2, 4, 6, 16)
         for BH in (1, 3) for P in (1, 4, 16, 152)]


@pytest.mark.parametrize("mode,causal,n,BH,P", CASES)
def test_generator_matches_simulator(mode, causal, n, BH, P):
    try:
        d.check_mode(mode, n, causal)
    except d.ScheduleError:
        assert dash.dash_schedule_num_tasks(BH, n, causal, mode) == -1
        with pytest.raises(dash.DashError) as ei:
            dash.dash_build_schedule(BH, n, causal, mode, P)
        assert ei.value.code == 2
        return
    for c, r in ((4, 1), (1, 3), (7, 2)):
        try:
            py = d.schedule_tables(mode, BH, n, causal, P, c, r)
        except d.Deadlock:
            with pytest.raises(dash.DashError) as ei:
                dash.dash_build_schedule(BH, n, causal, mode, P, c, r)
            assert ei.value.code == 6
            continue
        tasks, off, ms = dash.dash_build_schedule(BH, n, causal, mode, P, c, r)
        np.testing.assert_array_equal(tasks, np.asarray(py[0], dtype=np.int32).reshape(-1, 4))
        np.testing.assert_array_equal(off, np.asarray(py[1], dtype=np.int32))
        assert ms == py[2]


@pytest.mark.parametrize("BH,n,causal,mode", [(64, 16, True, "symmetric_shift"), (32, 32, False, "shift"),
                                              (32, 64, True, "descending_q"), (16, 128, True, "serial")])
def test_generator_matches_simulator_at_full_size(BH, n, causal, mode):
    py = d.schedule_tables(mode, BH, n, causal, 152)
    tasks, off, ms = dash.dash_build_schedule(BH, n, causal, mode, 152)
    np.testing.assert_array_equal(tasks, np.asarray(py[0], dtype=np.int32).reshape(-1, 4))
    np.testing.assert_array_equal(off, np.asarray(py[1], dtype=np.int32))
    assert ms == py[2]


@pytest.mark.parametrize("BH,n,causal,mode", [(8, 4, False, "shift"), (6, 8, True, "symmetric_shift"),
                                              (4, 6, True, "descending_q")])
def test_cta_choice_is_best_simulated(BH, n, causal, mode):
    P_max = 40
    chosen = dash.dash_choose_ctas(BH, n, causal, mode, P_max)
    gang = n // 2 if mode == "symmetric_shift" else n
    top = min(P_max, BH * gang)
    cyclic = mode == "shift"   # only shift is restricted to whole gangs
    mults = [m for m in range((top // gang) * gang, gang - 1, -gang)]
    cands = mults[:16] if cyclic else ([top] + [m for m in mults if m != top][:15])
    spans = {}
    for P in cands:
        try:
            spans[P] = d.simulate(d.all_chains(mode, BH, n, causal), P, 4, 1).makespan
        except d.Deadlock:
            pass
    best = min(spans.values())
    assert chosen == min(P for P, s in spans.items() if s == best)


def test_error_codes_without_gpu():
    # argument checks run before any CUDA call
    L = dash.lib()
    import ctypes
    nul = ctypes.c_void_p(0)
    assert L.dash_attn_bwd(*([nul] * 9), 1, 1, 128, 96, 0, 0.1, 1, nul) == 2      # D = 96
    assert L.dash_attn_bwd(*([nul] * 9), 1, 1, 128, 64, 0, -1.0, 1, nul) == 1     # scale <= 0
    assert L.dash_attn_bwd(*([nul] * 9), -1, 1, 128, 64, 0, 0.1, 1, nul) == 1    # B < 0
    assert L.dash_attn_bwd(*([nul] * 9), 0, 1, 128, 64, 0, 0.1, 1, nul) == 0     # empty: no-op
    assert L.dash_attn_fwd(*([nul] * 5), 1, 1, 128, 64, 0, float("nan"), nul) == 1
    assert "scale" in dash.dash_last_error()
    assert dash.dash_schedule_num_tasks(2, 8, True, "shift") == -1
    assert dash.dash_schedule_num_tasks(2, 8, True, "serial") == 2 * 36
    assert dash.dash_schedule_num_tasks(2, 7, True, "symmetric_shift") == -1
    # dq_chains other than 0, 1, 2 is rejected before any CUDA call
    fake = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced
    opt = dash.BwdOptions(0, 0, 0, 0, 0, None, None, None, None, None, 3)
    assert L.dash_attn_bwd_ex(*([fake] * 9), 1, 1, 128, 64, 0, 0.1, 1, ctypes.byref(opt), nul) == 1
    assert "dq_chains" in dash.dash_last_error()
    # split gangs: a k that does not divide the gang, a negative k, and k with fill or die-aware placement
    # (S = 1024, tile 128: a shift gang of 8 chains) are rejected before any CUDA call
    for fields, code, words in [({"shift_split": 3}, 2, "divide"), ({"shift_split": -2}, 1, "shift_split"),
                                ({"shift_split": 2, "shift_fill": 1}, 2, "without fill"),
                                ({"shift_split": 2, "die_aware": 1}, 2, "split gangs"),
                                ({"rank_order": 2}, 1, "rank_order"),
                                ({"rank_order": 1, "shift_fill": 1}, 2, "rank_order"),
                                ({"rank_order": 1, "die_aware": 1}, 2, "rank_order")]:
        opt = dash.BwdOptions()
        for f, x in fields.items():
            setattr(opt, f, x)
        opt.tile = 128
        assert L.dash_attn_bwd_ex(*([fake] * 9), 1, 1, 1024, 64, 0, 0.1, 3, ctypes.byref(opt), nul) == code
        assert words in dash.dash_last_error()
    # more tasks than the 32-bit task tables index: 2^16 heads at S = 2^20 (full mask, n = 8192)
    assert L.dash_attn_bwd(*([fake] * 9), 1, 1 << 16, 1 << 20, 64, 0, 0.1, 1, nul) == 2
    assert "32-bit" in dash.dash_last_error()
    # and a causal one of 2^12 heads (1.4e11 tasks)
    assert L.dash_attn_bwd(*([fake] * 9), 1, 1 << 12, 1 << 20, 64, 1, 0.1, 1, nul) == 2


@pytest.mark.parametrize("BH,n,causal,c,r", [(8, 4, False, 4, 1), (8, 4, False, 1, 4), (6, 8, True, 4, 1),
                                             (6, 8, True, 1, 3), (4, 6, True, 4, 1), (3, 5, False, 2, 2),
                                             (32, 16, True, 4, 1)])
def test_schedule_choice_is_best_simulated(BH, n, causal, c, r):
    # the runtime choice: smallest simulated makespan over the deterministic
    # schedules valid for the mask, each at its chosen CTA count
    P_max = 40
    spans = {}
    for mode in ("serial", "descending_q", "shift", "symmetric_shift"):
        if (mode == "shift" and causal) or (mode == "symmetric_shift" and (not causal or n % 2)):
            continue
        P = dash.dash_choose_ctas(BH, n, causal, mode, P_max, c, r)
        spans[mode] = (d.simulate(d.all_chains(mode, BH, n, causal), P, c, r).makespan, P)
    best = min(s for s, _ in spans.values())
    want = next(m for m in ("serial", "descending_q", "shift", "symmetric_shift") if m in spans and spans[m][0] == best)
    assert dash.dash_choose_schedule(BH, n, causal, P_max, c, r) == (want, spans[want][1], best)


@pytest.mark.parametrize("BH,n,causal,c,r", [(8, 4, False, 4, 1), (6, 8, True, 4, 1), (6, 8, True, 1, 3),
                                             (3, 12, False, 2, 2), (16, 16, True, 4, 1)])
def test_schedule_choice_with_split_gangs(BH, n, causal, c, r):
    # the split-aware runtime choice: shift / symmetric shift enter with the split and CTA count that
    # dash_choose_split picks (its makespan re-simulated by the oracle), the others as in dash_choose_schedule
    P_max = 30
    spans = {}
    for mode in ("serial", "descending_q", "shift", "symmetric_shift"):
        if (mode == "shift" and causal) or (mode == "symmetric_shift" and (not causal or n % 2)):
            continue
        if mode in ("shift", "symmetric_shift"):
            k, P, ms = dash.dash_choose_split(BH, n, causal, mode, P_max, 0, c, r)
            assert ms == d.simulate(d.split_chains(mode, BH, n, causal, k), P, c, r).makespan
            spans[mode] = (ms, P, k)
        else:
            P = dash.dash_choose_ctas(BH, n, causal, mode, P_max, c, r)
            spans[mode] = (d.simulate(d.all_chains(mode, BH, n, causal), P, c, r).makespan, P, 1)
    best = min(s for s, _, _ in spans.values())
    want = next(m for m in ("serial", "descending_q", "shift", "symmetric_shift") if m in spans and spans[m][0] == best)
    assert dash.dash_choose_schedule_split(BH, n, causal, P_max, c, r) == (want, spans[want][1], spans[want][2], best)
    # never worse than the choice without split gangs
    assert best <= dash.dash_choose_schedule(BH, n, causal, P_max, c, r)[2]


FILL_CASES = [("shift", False, 32, 32, 152), ("shift", False, 12, 16, 152), ("shift", False, 4, 32, 152),
              ("shift", False, 48, 16, 152), ("shift", False, 7, 4, 10), ("shift", False, 5, 3, 7),
              ("shift", False, 9, 6, 20), ("shift", False, 16, 8, 20), ("shift", False, 16, 128, 152),
              ("symmetric_shift", True, 32, 64, 152), ("symmetric_shift", True, 64, 16, 152),
              ("symmetric_shift", True, 9, 8, 14), ("symmetric_shift", True, 5, 6, 11),
              ("symmetric_shift", True, 16, 8, 10), ("symmetric_shift", True, 16, 128, 152)]


@pytest.mark.parametrize("mode,causal,BH,n,P", FILL_CASES)
def test_fill_generator_matches_simulator(mode, causal, BH, n, P):
    for c, r in ((4, 1),) if n >= 64 else ((4, 1), (1, 1), (1, 3)):   # the pure-Python simulator is slow at large n
        py_tasks, py_off, py_ms, py_hs, py_fill = d.fill_tables(mode, BH, n, causal, P, c, r)
        tasks, off, Pc, hs, fill, ms = dash.dash_build_shift_fill(BH, n, causal, mode, P, c, r)
        np.testing.assert_array_equal(tasks, np.asarray(py_tasks, dtype=np.int32).reshape(-1, 4))
        np.testing.assert_array_equal(off, np.asarray(py_off, dtype=np.int32))
        assert (Pc, hs, fill, ms) == (len(py_off) - 1, py_hs, py_fill, py_ms)


def test_fill_rejections():
    with pytest.raises(d.Deadlock):
        d.fill_tables("shift", 3, 8, False, 5)
    with pytest.raises(dash.DashError) as ei:
        dash.dash_build_shift_fill(3, 8, False, "shift", 5)
    assert ei.value.code == 6
    with pytest.raises(dash.DashError) as ei:   # fill applies to the cyclic schedules only
        dash.dash_build_shift_fill(4, 8, False, "serial", 40)
    assert ei.value.code == 2
    import ctypes
    fake = ctypes.c_void_p(1 << 20)
    opt = dash.BwdOptions(0, 0, 0, 0, 0, None, None, None, None, None, 0, 2)
    assert dash.lib().dash_attn_bwd_ex(*([fake] * 9), 1, 1, 128, 64, 0, 0.1, 3, ctypes.byref(opt),
                                       ctypes.c_void_p(0)) == 1
    assert "shift_fill" in dash.dash_last_error()


@pytest.mark.parametrize("BH,n,causal,P", [(8, 4, False, 10), (6, 8, True, 12), (4, 6, True, 40), (12, 16, False, 152)])
def test_cost_fit_recovers_simulated_costs(BH, n, causal, P):
    # fed the simulator's own makespans as "measured" times, the fit returns
    # the r that produced them, and the C++ fit equals the oracle's
    for r0 in (1, 3, 8, 24, 64, 256):
        a = d.simulate(d.all_chains("atomic", BH, n, causal), min(P, BH * n), 8, r0, ordered=False).makespan
        s = d.simulate(d.all_chains("serial", BH, n, causal), min(P, BH * n), 8, r0).makespan
        assert dash.dash_fit_costs(BH, n, causal, P, 0.01 * a, 0.01 * s) == (8, r0)
        assert d.fit_costs(BH, n, causal, P, 0.01 * a, 0.01 * s) == (8, r0)
    for ta, ts in ((1.0, 1.0), (1.0, 1.7), (2.0, 9.0), (1.0, 0.5)):
        assert dash.dash_fit_costs(BH, n, causal, P, ta, ts) == d.fit_costs(BH, n, causal, P, ta, ts)


def test_cost_fit_rejects_bad_arguments():
    for args in ((0, 4, False, 10, 1.0, 1.0), (4, 4, False, 10, 0.0, 1.0), (4, 4, False, 10, 1.0, float("nan"))):
        with pytest.raises(dash.DashError) as ei:
            dash.dash_fit_costs(*args)
        assert ei.value.code == 1


def _finishes(tasks, off, chains):
    """Plain reference for the table check: repeat passes over the CTAs, letting each
    perform its next add when the previous position of its chain is done."""
    nxt, ptr = {}, list(off[:-1])
    moved = True
    while moved:
        moved = False
        for s in range(len(off) - 1):
            while ptr[s] < off[s + 1]:
                bh, kv, q, w = (int(x) for x in tasks[ptr[s]])
                rank = w & dash.TASK_RANK_MASK
                key = (bh, q, rank % chains)
                if nxt.get(key, 0) != rank // chains:
                    break
                nxt[key] = rank // chains + 1
                ptr[s] += 1
                moved = True
    return all(ptr[s] == off[s + 1] for s in range(len(off) - 1))


def test_table_check_accepts_generated_tables():
    for mode, causal, n in (("serial", False, 4), ("descending_q", True, 5), ("shift", False, 4),
                            ("symmetric_shift", True, 6)):
        for P in (3, 8, 40):
            try:
                t, off, _ = dash.dash_build_schedule(3, n, causal, mode, P)
            except dash.DashError:
                continue
            for chains in (0, 2):
                dash.dash_check_table(3, n, causal, t, off, chains)


def test_table_check_rejects_gaps_repeats_and_cycles():
    F, L = dash.TASK_FIRST, dash.TASK_LAST
    bad = {
        # KV 0 adds to Q tile 0 at rank 1 before Q tile 1 at rank 0; KV 1 the other way round
        "cycle": ([[0, 0, 0, 1 | F], [0, 0, 1, 0 | L], [0, 1, 1, 1 | F], [0, 1, 0, 0 | L]], [0, 2, 4], 2),
        "gap": ([[0, 0, 0, 0 | F | L], [0, 2, 0, 2 | F | L]], [0, 1, 2], 3),
        "repeats": ([[0, 0, 0, 0 | F | L], [0, 1, 0, 0 | F | L]], [0, 1, 2], 2),
    }
    for word, (t, off, n) in bad.items():
        with pytest.raises(dash.DashError) as ei:
            dash.dash_check_table(1, n, False, np.array(t, dtype=np.int32), off)
        assert ei.value.code == 6 and word in dash.dash_last_error(), dash.dash_last_error()


@pytest.mark.parametrize("seed", range(4))
def test_table_check_agrees_with_a_plain_run(seed):
    # random tables: each CTA runs one KV tile over the Q tiles in a random
    # order; each dQ tile's ranks are a random permutation of its KV tiles
    rng = np.random.default_rng(seed)
    verdicts = set()
    for _ in range(150):
        n, BH = int(rng.integers(2, 5)), int(rng.integers(1, 3))
        chains = int(rng.integers(1, 3))
        ranks = {(bh, q): rng.permutation(n) for bh in range(BH) for q in range(n)}
        tasks, off = [], [0]
        for bh in range(BH):
            for kv in range(n):
                order = rng.permutation(n)
                for j, q in enumerate(order):
                    w = int(ranks[(bh, q)][kv]) | (dash.TASK_FIRST if j == 0 else 0) | \
                        (dash.TASK_LAST if j == n - 1 else 0)
                    tasks.append([bh, kv, int(q), w])
                off.append(len(tasks))
        tasks = np.array(tasks, dtype=np.int32)
        ok = _finishes(tasks, off, chains)
        verdicts.add(ok)
        if ok:
            dash.dash_check_table(BH, n, False, tasks, off, chains)
        else:
            with pytest.raises(dash.DashError) as ei:
                dash.dash_check_table(BH, n, False, tasks, off, chains)
            assert ei.value.code == 6
    assert verdicts == {True, False}


def test_schedule_choice_rejects_bad_arguments():
    with pytest.raises(dash.DashError):
        dash.dash_choose_schedule(0, 4, False, 40)
    assert "dash_choose_schedule" in dash.dash_last_error()


@pytest.mark.parametrize("mode,causal,BH,n", [("shift", False, 3, 8), ("shift", False, 2, 16), ("symmetric_shift", True, 3, 8),
                                              ("symmetric_shift", True, 2, 16)])
@pytest.mark.parametrize("split", [1, 2, 4])
def test_split_generator_matches_simulator(mode, causal, BH, n, split):
    gang = n if mode == "shift" else n // 2
    for P in (gang // split, 2 * gang // split + 1, 40):
        for c, r in ((4, 1), (2, 3)):
            py_tasks, py_off, py_ms = d.split_tables(mode, BH, n, causal, split, P, c, r)
            tasks, off, ms = dash.dash_build_split_schedule(BH, n, causal, mode, split, P, c, r)
            assert np.array_equal(tasks, np.asarray(py_tasks, dtype=np.int32).reshape(-1, 4))
            assert np.array_equal(off, np.asarray(py_off, dtype=np.int32)) and ms == py_ms


def test_split_rejections_and_cta_choice():
    with pytest.raises(dash.DashError) as ei:   # split gangs apply to the cyclic schedules only
        dash.dash_build_split_schedule(2, 8, False, "serial", 2, 8)
    assert ei.value.code == 2
    with pytest.raises(dash.DashError) as ei:   # 3 does not divide a gang of 8
        dash.dash_build_split_schedule(2, 8, False, "shift", 3, 8)
    assert ei.value.code == 2
    assert dash.dash_choose_split_ctas(2, 8, False, "shift", 3, 40) == -1
    # the CTA count is a multiple of the sub-gang, chosen by simulated makespan
    for split in (1, 2, 4):
        P = dash.dash_choose_split_ctas(32, 32, False, "shift", split, 152, 8, 512)
        assert P % (32 // split) == 0 and P <= 152
        spans = {}
        for cand in range(32 // split, 153, 32 // split):
            spans[cand] = d.simulate(d.split_chains("shift", 32, 32, False, split), cand, 8, 512).makespan
        best = min(spans.values())
        assert spans[P] == best and P == min(c for c, s in spans.items() if s == best)


@pytest.mark.parametrize("BH,n,causal,mode,P_max", [(4, 8, False, "shift", 20), (3, 12, False, "shift", 30),
                                                    (6, 8, True, "symmetric_shift", 12),
                                                    (5, 12, True, "symmetric_shift", 14),
                                                    (16, 16, True, "symmetric_shift", 30)])   # a tie: k = 2 on 28
def test_split_choice_is_best_simulated(BH, n, causal, mode, P_max):
    # shift_split = -1: every k dividing the gang, k = 1 on up to sixteen candidate CTA counts and k > 1 on
    # its two largest (multiples of the sub-gang; symmetric shift also P_max itself), each simulated by the
    # oracle; smallest makespan, ties to fewer CTAs within a k, then across k to a sub-gang that divides its
    # CTA count, then to the smaller k
    gang = n // 2 if causal else n
    top = min(P_max, BH * gang)
    best = None
    for k in [k for k in range(1, gang + 1) if gang % k == 0]:
        g = gang // k
        cands = [] if mode == "shift" else [top]
        m = (top // g) * g
        while m >= g and len(cands) < (16 if k == 1 else 2):
            if mode == "shift" or m != top:
                cands.append(m)
            m -= g
        spans = []
        for P in cands:
            try:
                spans.append((d.simulate(d.split_chains(mode, BH, n, causal, k), P, 4, 1).makespan, P))
            except d.Deadlock:
                continue
        if spans:
            ms, P = min(spans)
            key = (ms, P % g != 0, k)
            if best is None or key < best[0]:
                best = (key, P)
    k, P, ms = dash.dash_choose_split(BH, n, causal, mode, P_max)
    assert (ms, P % ((n // 2 if causal else n) // k) != 0, k) == best[0] and P == best[1]
    # on a given CTA count, shift only takes the k whose sub-gang divides it
    k2, P2, _ = dash.dash_choose_split(BH, n, causal, mode, P_max, num_ctas=P_max)
    assert P2 == P_max and (mode != "shift" or P_max % (gang // k2) == 0)
    assert dash.dash_choose_split(BH, n, causal, "serial", P_max)[0] == -1


TIMED_CASES = [("shift", False, 3, 8, 1), ("shift", False, 5, 4, 1), ("shift", False, 3, 8, 2), ("shift", False, 2, 12, 2),
               ("symmetric_shift", True, 3, 8, 1), ("symmetric_shift", True, 2, 12, 2), ("serial", False, 3, 8, 1),
               ("serial", True, 5, 4, 1), ("descending_q", True, 2, 12, 1), ("atomic", False, 3, 8, 1)]


@pytest.mark.parametrize("mode,causal,BH,n,split", TIMED_CASES)
def test_timed_generator_matches_simulator(mode, causal, BH, n, split):
    # timed ranks (an extension): the C++ tables equal the oracle twin's, whole or split gangs, on CTA counts
    # that are and are not multiples of the gang; atomic keeps its own (unordered) table
    for P in (3, 7, 10, 16, 40):
        for c, r in ((4, 1), (2, 3)):
            tasks, off, ms = dash.dash_build_schedule_ex(BH, n, causal, mode, split, 1, P, c, r)
            if mode == "atomic":
                py = d.schedule_tables(mode, BH, n, causal, P, c, r)
            else:
                py = d.timed_tables(mode, BH, n, causal, P, split, c, r)
            assert np.array_equal(tasks, np.asarray(py[0], dtype=np.int32).reshape(-1, 4))
            assert np.array_equal(off, np.asarray(py[1], dtype=np.int32)) and ms == py[2]


def test_timed_ranks_rejections():
    with pytest.raises(dash.DashError) as ei:
        dash.dash_build_schedule_ex(2, 8, False, "shift", 1, 2, 8)
    assert ei.value.code == 1
    with pytest.raises(dash.DashError) as ei:   # a split of the serial schedule
        dash.dash_build_schedule_ex(2, 8, False, "serial", 2, 1, 8)
    assert ei.value.code == 2


@pytest.mark.parametrize("BH,n,causal,c,r", [(8, 4, False, 4, 1), (5, 8, False, 4, 1), (6, 8, True, 4, 1),
                                             (6, 8, True, 1, 3), (16, 16, True, 4, 1), (3, 12, False, 2, 2)])
def test_layout_choice_is_best_simulated(BH, n, causal, c, r):
    # every layout priced by the oracle simulator: each ordered schedule in its own order on its chosen CTA count,
    # the cyclic schedule with the chosen split, and each with timed ranks; ties keep the first candidate
    P_max = 30
    cands = []
    for mode in ("serial", "descending_q", "shift", "symmetric_shift"):
        if (mode == "shift" and causal) or (mode == "symmetric_shift" and (not causal or n % 2)):
            continue
        cyclic = mode in ("shift", "symmetric_shift")
        P = dash.dash_choose_ctas(BH, n, causal, mode, P_max, c, r)
        cands.append((d.simulate(d.all_chains(mode, BH, n, causal), P, c, r).makespan, mode, P, 1, 0))
        k, Pk, _ = dash.dash_choose_split(BH, n, causal, mode, P_max, 0, c, r) if cyclic else (1, 0, 0)
        if k > 1:
            cands.append((d.simulate(d.split_chains(mode, BH, n, causal, k), Pk, c, r).makespan, mode, Pk, k, 0))
        gang = n // 2 if mode == "symmetric_shift" else n
        Pall = min(P_max, BH * gang)
        cands.append((d.timed_tables(mode, BH, n, causal, Pall, 1, c, r)[2], mode, Pall, 1, 1))
        if k > 1:
            cands.append((d.timed_tables(mode, BH, n, causal, Pk, k, c, r)[2], mode, Pk, k, 1))
    best = min(cands, key=lambda x: x[0])   # min keeps the first of equal makespans
    name, P, k, ro, ms = dash.dash_choose_layout(BH, n, causal, P_max, c, r)
    assert (ms, name, P, k, ro) == best

