"""Cluster hand-offs on the GPU (dash_bwd_options_t.cluster_size).

With clusters, a rank whose predecessor runs in the same cluster takes its
turn from a shared-memory counter instead of the global semaphore.  The ranks
and adds do not change, so every ordered schedule must give the same bits with
clusters as without, and meet the oracle."""
import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash
import workloads
from oracle import attention as A

from _gpu import Problem, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("S,D,causal,sched,chains", [(1024, 128, False, "shift", 1), (1024, 128, True, "symmetric_shift", 1),
                                                     (1024, 64, False, "serial", 1), (1024, 64, True, "descending_q", 1),
                                                     (1024, 128, False, "shift", 2), (700, 128, True, "serial", 2)])
def test_clusters_give_the_same_bits_and_meet_the_oracle(S, D, causal, sched, chains):
    P = Problem(2, 4, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    plain = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, dq_chains=chains, cluster_size=1)
    for size in (2, 4):
        try:
            got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, dq_chains=chains, cluster_size=size)
        except dash.DashError as e:   # clusters of 4 need a CTA count that 4 divides
            assert size == 4 and e.code == 2
            continue
        dash.dash_sync_status()
        for name, a, b in zip(("dQ", "dK", "dV"), got, plain):
            assert torch.equal(a, b), f"{sched} with clusters of {size}: {name} differs"
    q, k, v, do = P.f64
    ro, rl = A.forward(q, k, v, causal, P.scale)
    for name, x, r in zip(("dQ", "dK", "dV"), got, A.backward(q, k, v, ro, do, rl, causal, P.scale)):
        assert_close(f"{sched} clustered {name}", x, r)


@pytest.mark.parametrize("wname,sched", [("full_s4096_d128", "shift"), ("causal_s16384_d128", "symmetric_shift"),
                                         ("causal_s8192_d64", "descending_q")])
def test_clusters_full_size_same_bits(wname, sched):
    w = workloads.WORKLOADS[wname]
    q, k, v, do = (t.cuda() for t in workloads.make_workload_inputs(w))
    o, lse = dash.attn_fwd(q, k, v, w.causal, w.scale)
    plain = dash.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, sched, tile=w.tile, cluster_size=1)
    got = dash.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, sched, tile=w.tile, cluster_size=2)
    dash.dash_sync_status()
    for name, a, b in zip(("dQ", "dK", "dV"), got, plain):
        assert torch.equal(a, b), f"{wname} {sched}: {name} differs with clusters"


def test_cluster_size_that_does_not_divide_is_refused():
    P = Problem(1, 3, 512, 128, False)   # shift: 12 chains on 12 CTAs: clusters of 8 do not divide
    o, lse = dash.attn_fwd(P.q, P.k, P.v, False, P.scale)
    with pytest.raises(dash.DashError) as ei:
        dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, False, P.scale, "shift", cluster_size=8)
    assert ei.value.code == 2
