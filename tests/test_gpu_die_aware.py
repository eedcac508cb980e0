"""Die-aware placement on the GPU (dash_bwd_options_t.die_aware, an extension).

The placement changes where each chain runs and where each dQ semaphore
lives, never the tasks, their ranks or the adds, so the results must be the
plain schedule's bits.  The traced kernel then shows that every whole gang of
a shift schedule ran on SMs of one group of the measured die map.
"""
import numpy as np
import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash
import workloads
from deterministic_attention_backward_fa_gb300 import trace as T

from _gpu import Problem, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def test_die_map_has_two_groups():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    g, n0, n1 = dash.dash_die_map()
    assert n0 + n1 == sms and n0 >= 8 and n1 >= 8
    assert int((g >= 0).sum()) == sms


@pytest.mark.parametrize("S,D,causal,sched,chains", [(512, 128, False, "shift", 1), (1024, 64, True, "symmetric_shift", 1),
                                                     (512, 128, False, "shift", 2)])
def test_die_aware_equals_plain_and_oracle(S, D, causal, sched, chains):
    P = Problem(2, 3, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    plain = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, dq_chains=chains)
    for _ in range(3):
        placed = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, dq_chains=chains, die_aware=1)
        dash.dash_sync_status()
        for name, a, b in zip(("dQ", "dK", "dV"), placed, plain):
            assert torch.equal(a, b), f"die-aware {sched} {name} differs from the plain schedule"
    q, k, v, do = P.f64
    from oracle import attention as A
    ro, rl = A.forward(q, k, v, causal, P.scale)
    for name, x, r in zip(("dQ", "dK", "dV"), placed, A.backward(q, k, v, ro, do, rl, causal, P.scale)):
        assert_close(f"die-aware {sched} {name}", x, r)


@pytest.mark.parametrize("wname,sched", [("full_s4096_d128", "shift"), ("causal_s8192_d64", "symmetric_shift")])
def test_die_aware_full_size_gangs_on_one_group(wname, sched):
    w = workloads.WORKLOADS[wname]
    q, k, v, do = (t.cuda() for t in workloads.make_workload_inputs(w))
    o, lse = dash.attn_fwd(q, k, v, w.causal, w.scale)
    plain = dash.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, sched, tile=w.tile)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    BH, n = w.B * w.H, w.n_blocks
    tasks, off, ctas = T.task_table(BH, n, w.causal, sched, sms)
    tr = torch.zeros((len(tasks), dash.TRACE_SLOTS), dtype=torch.int64, device="cuda")
    outs = [torch.empty_like(q) for _ in range(3)]
    dash.dash_attn_bwd_ex(q, k, v, o, do, lse, *outs, w.causal, w.scale, sched, tile=w.tile, trace=tr, die_aware=1)
    dash.dash_sync_status()
    for name, a, b in zip(("dQ", "dK", "dV"), outs, plain):
        assert torch.equal(a, b), f"die-aware {name} differs from the plain schedule at full size"
    tr = tr.cpu().numpy()
    groups, _, _ = dash.dash_die_map()
    meta = tr[:, T.META]
    slot_sm = {int(m) & 0xFFFF: int(m) >> 16 for m in meta}
    assert set(slot_sm) == {c for c in range(ctas) if off[c + 1] > off[c]}
    gang = n if sched == "shift" else n // 2
    for c in range(ctas):   # each slot's tasks are in its own rows of the table
        assert all((int(m) & 0xFFFF) == c for m in meta[off[c]:off[c + 1]])
    whole = ctas // gang if sched == "shift" else 0
    for g0 in range(0, whole * gang, gang):
        grp = {int(groups[slot_sm[s]]) for s in range(g0, g0 + gang) if s in slot_sm}
        assert len(grp) == 1, f"gang at slots {g0}.. ran on both groups of SMs"
