"""Host half of the die-aware placement (an extension for the shift schedules).

The clustering must recover a planted two-die structure from noisy L2
latencies (SM groups and line homes, up to the naming of the groups), and the
placement tables must keep every whole gang of chains on one group of SMs,
give every slot exactly one SM, and home each dQ tile's semaphore on the group
that runs the tile's adds.  No GPU needed.
"""
import numpy as np
import pytest

import deterministic_attention_backward_fa_gb300 as dash


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _planted(n_sms, n_lines, gap, noise, seed):
    rng = np.random.default_rng(seed)
    grp = rng.integers(0, 2, n_sms)
    grp[0], grp[1] = 0, 1
    home = rng.integers(0, 2, n_lines)
    lat = 270 + gap * (grp[:, None] != home[None, :]) + rng.integers(-noise, noise + 1, (n_sms, n_lines))
    return lat.astype(np.uint32), grp, home


@pytest.mark.parametrize("n_sms,n_lines,gap,noise,seed", [(152, 4096, 33, 12, 0), (20, 300, 40, 5, 1),
                                                           (2, 64, 30, 3, 2)])
def test_clustering_recovers_planted_dies(n_sms, n_lines, gap, noise, seed):
    lat, grp, home = _planted(n_sms, n_lines, gap, noise, seed)
    g, h = dash.dash_cluster_latencies(lat)
    swap = g[0] != grp[0]          # group names are arbitrary: compare up to a swap
    if swap:
        g, h = 1 - g, 1 - h
    assert np.array_equal(g, grp)
    assert np.array_equal(h, home)


def test_clustering_rejects_too_few_sms():
    with pytest.raises(dash.DashError) as ei:
        dash.dash_cluster_latencies(np.full((1, 8), 270, dtype=np.uint32))
    assert ei.value.code == 1


def _group_of(smids):
    out = {}
    for g, lst in enumerate(smids):
        for s in lst:
            out[int(s)] = g
    return out


@pytest.mark.parametrize("BH,n,mode,P,n0,n1", [(4, 4, "shift", 16, 10, 10), (8, 8, "shift", 32, 20, 17),
                                               (6, 8, "symmetric_shift", 20, 12, 12)])
def test_placement_keeps_gangs_on_one_group(BH, n, mode, P, n0, n1):
    causal = mode == "symmetric_shift"
    tasks, off, _ = dash.dash_build_schedule(BH, n, causal, mode, P)
    gang = n if mode == "shift" else n // 2
    rng = np.random.default_rng(P)
    ids = rng.permutation(200)[: n0 + n1]          # SM ids need not be contiguous
    smids = (sorted(ids[:n0]), sorted(ids[n0:]))
    lines = (list(range(0, 300, 2)), list(range(1, 300, 2)))
    slot_of, sem = dash.dash_place_schedule(tasks, off, gang, BH, n, 1, smids, lines, 199)
    gmap = _group_of(smids)
    slots = slot_of[slot_of >= 0]
    assert sorted(slots.tolist()) == list(range(P)), "every slot runs on exactly one SM"
    group_of_slot = {int(s): gmap[i] for i, s in enumerate(slot_of) if s >= 0}
    # in these cases every gang fits whole in the group with more SMs left
    for g0 in range(0, P - P % gang, gang):
        groups = {group_of_slot[s] for s in range(g0, g0 + gang)}
        assert len(groups) == 1, f"gang at slots {g0}.. spans both groups"
    assert len(set(sem.tolist())) == len(sem), "semaphores share a sector"
    assert all(x % 8 == 0 for x in sem), "semaphores sit on 32-byte sectors"
    # each tile's semaphore is homed on the group that runs most of the tile's adds
    home = {ln: g for g, lst in enumerate(lines) for ln in lst}
    votes = {}
    for c in range(P):
        for t in range(off[c], off[c + 1]):
            bh, _, q, _ = tasks[t]
            votes.setdefault((bh, q), [0, 0])[group_of_slot[c]] += 1
    for (bh, q), v in votes.items():
        want = 1 if v[1] > v[0] else 0
        assert home[sem[bh * n + q] // 32] == want


def test_placement_fails_without_enough_sms_or_lines():
    tasks, off, _ = dash.dash_build_schedule(2, 4, False, "shift", 8)
    with pytest.raises(dash.DashError) as ei:
        dash.dash_place_schedule(tasks, off, 4, 2, 4, 1, ([0, 1, 2], [3, 4]), ([0], [1]), 10)
    assert ei.value.code == 6
    with pytest.raises(dash.DashError) as ei:   # head 1's four semaphores belong on group 1, which has no line
        dash.dash_place_schedule(tasks, off, 4, 2, 4, 1, (list(range(4)), list(range(4, 8))), ([0], []), 10)
    assert ei.value.code == 6
