"""The trace tool's summary on a synthetic trace (no GPU): the hop of each dQ
chain is measured from the predecessor's release to the successor's turn in
the table's rank order, and a rank that took its turn before its
predecessor's release began is counted as a violation of the order."""
import numpy as np
import pytest

import deterministic_attention_backward_fa_gb300 as dash
from deterministic_attention_backward_fa_gb300 import trace as T


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _synthetic(tasks, hop_ns=100):
    """Stamps in which rank k of each tile takes its turn hop_ns after rank k - 1 began its release."""
    n_tasks = len(tasks)
    tr = np.zeros((n_tasks, dash.TRACE_SLOTS), dtype=np.int64)
    rank = tasks[:, 3] & ((1 << 24) - 1)
    order = np.lexsort((rank, tasks[:, 2], tasks[:, 0]))   # by head, tile, rank
    t_ns = 1000
    prev_key = None
    for t in order:
        key = (tasks[t, 0], tasks[t, 2])
        if key != prev_key:
            t_ns += 10000
            prev_key = key
        tr[t, T.ACQ0] = t_ns - 50
        tr[t, T.ACQ1] = t_ns
        tr[t, T.REL0] = t_ns + 400
        tr[t, T.REL1] = t_ns + 450
        t_ns += 400 + hop_ns
    for t in range(n_tasks):
        tr[t, T.MMA_DP:T.MMA_END + 1] = [10 * t + 1, 10 * t + 2, 10 * t + 3, 10 * t + 4]
        tr[t, T.CLK_AT_ACQ0] = tr[t, T.ACQ0] * 2   # a 2 GHz clock on the same axis
    return tr


def test_summary_measures_hops_and_finds_no_violation():
    tasks, off, _ = dash.dash_build_schedule(2, 4, False, "shift", 8)
    tr = _synthetic(tasks)
    rows, mhz, viol, _ = T.summarize(tasks, off, tr, chains=1)
    assert viol == 0
    got = dict(rows)
    assert got["hop: predecessor's release starts until this rank's turn is taken, ns"].startswith("100 ")
    assert got["hop: predecessor's release returned until this rank's turn is taken, ns"].startswith("50 ")
    assert got["release store (its fence waits for the adds), ns"].startswith("50 ")
    assert abs(mhz - 2000.0) < 1e-6


def test_summary_counts_a_rank_that_jumped_its_turn():
    tasks, off, _ = dash.dash_build_schedule(2, 4, True, "symmetric_shift", 4)
    tr = _synthetic(tasks)
    rank = tasks[:, 3] & ((1 << 24) - 1)
    t = int(np.nonzero(rank == 2)[0][0])       # a rank-2 task: make it take its turn far too early
    tr[t, T.ACQ1] = 0
    _, _, viol, _ = T.summarize(tasks, off, tr, chains=1)
    assert viol == 1
