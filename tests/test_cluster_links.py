"""Cluster hand-offs of the dQ order (dash_bwd_options_t.cluster_size), host half.

A linked rank takes its turn from a counter that its predecessor's CTA raises
in the same cluster, one counter per producing CTA.  The links must stay
inside a cluster, join exactly the consecutive ranks of a dQ tile's order,
and, per (producer, consumer) pair, be taken in the order they are given, so
that counting arrivals is enough.  A replay of the table in which linked turns
wait on such counters must then finish with every tile's adds in rank order.
"""
import collections

import numpy as np
import pytest

import deterministic_attention_backward_fa_gb300 as dash


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _check_links(tasks, off, C, BH, n, chains, links):
    P = len(off) - 1
    cta = np.zeros(len(tasks), dtype=int)
    for c in range(P):
        cta[off[c]:off[c + 1]] = c
    rank = tasks[:, 3] & ((1 << 24) - 1)
    order = collections.defaultdict(list)
    for t in range(len(tasks)):
        order[(tasks[t, 0], tasks[t, 2], rank[t] % chains)].append((rank[t] // chains, t))
    pred = {}
    for v in order.values():
        v.sort()
        for (_, tp), (_, tc) in zip(v, v[1:]):
            pred[tc] = tp
    pairs = collections.defaultdict(list)
    for t in range(len(tasks)):
        w = int(links[t]) & 0xFFFFFFFF
        if w & (1 << 30):                        # takes its turn through a counter
            tp = pred[t]
            assert cta[tp] // C == cta[t] // C, "a link leaves its cluster"
            assert ((w >> 16) & 0xF) == cta[tp] % C
            wp = int(links[tp]) & 0xFFFFFFFF
            assert wp >> 31 and ((wp >> 20) & 0xF) == cta[t] % C, "the predecessor does not raise the counter"
            pairs[(cta[tp], cta[t])].append((t, tp))
        if w >> 31:
            assert any(pred.get(tc) == t and (int(links[tc]) & (1 << 30)) for tc in range(len(tasks)))
    for lst in pairs.values():
        lst.sort()
        prods = [tp for _, tp in lst]
        assert prods == sorted(prods), "a consumer takes a producer's turns out of order"
    return cta, rank, pred


def _replay(tasks, off, chains, links, cta, rank, pred):
    """Event-driven run: a CTA does its tasks in order; a task waits for its predecessor's add, through the
    producer's counter when linked (the k-th linked turn from a producer needs that producer's k-th raise)."""
    P = len(off) - 1
    ptr = list(off[:-1])
    done = set()
    raised = collections.Counter()      # (producer CTA, consumer CTA) -> raises so far
    taken = collections.Counter()
    adds = collections.defaultdict(list)
    progress = True
    while progress:
        progress = False
        for c in range(P):
            while ptr[c] < off[c + 1]:
                t = ptr[c]
                w = int(links[t]) & 0xFFFFFFFF
                if t in pred:
                    tp = pred[t]
                    if w & (1 << 30):
                        if raised[(cta[tp], c)] <= taken[(cta[tp], c)]:
                            break
                    elif tp not in done:
                        break
                if w & (1 << 30):
                    taken[(cta[pred[t]], c)] += 1
                adds[(tasks[t, 0], tasks[t, 2], rank[t] % chains)].append(rank[t] // chains)
                done.add(t)
                if w >> 31:
                    succ = [tc for tc, tp in pred.items() if tp == t][0]
                    raised[(c, cta[succ])] += 1
                ptr[c] += 1
                progress = True
    assert all(ptr[c] == off[c + 1] for c in range(P)), "the replay stalled"
    for v in adds.values():
        assert v == list(range(len(v))), "adds out of rank order"


@pytest.mark.parametrize("mode,causal,BH,n,P,C,chains", [("shift", False, 8, 8, 16, 8, 1), ("shift", False, 4, 16, 32, 16, 1),
                                                         ("serial", False, 6, 8, 24, 8, 1), ("descending_q", True, 6, 8, 16, 4, 1),
                                                         ("symmetric_shift", True, 8, 8, 16, 4, 1), ("shift", False, 8, 8, 32, 8, 2),
                                                         ("serial", True, 5, 6, 12, 4, 2)])
def test_links_stay_in_cluster_and_keep_the_order(mode, causal, BH, n, P, C, chains):
    tasks, off, _ = dash.dash_build_schedule(BH, n, causal, mode, P)
    links, k = dash.dash_cluster_links(tasks, off, C, BH, n, chains)
    assert k > 0
    cta, rank, pred = _check_links(tasks, off, C, BH, n, chains, links)
    _replay(tasks, off, chains, links, cta, rank, pred)


def test_shift_with_whole_gangs_links_most_hops():
    # gangs of 16 chains on clusters of 16 CTAs: only the hop that wraps round each gang leaves the cluster
    BH, n = 8, 16
    tasks, off, _ = dash.dash_build_schedule(BH, n, False, "shift", 32)
    links, k = dash.dash_cluster_links(tasks, off, 16, BH, n, 1)
    hops = BH * n * (n - 1)
    assert k >= hops * (n - 1) // n


def test_no_links_without_clusters():
    tasks, off, _ = dash.dash_build_schedule(4, 4, False, "shift", 16)
    links, k = dash.dash_cluster_links(tasks, off, 1, 4, 4, 1)
    assert k == 0 and not links.any()
