"""The traced build of the main kernel (dash_bwd_options_t.trace).

Its stamps must not change the results (same bits as the plain kernel), every
task must be stamped, each role's stamps must come in program order, and, for
an ordered schedule, every rank of a dQ tile must take its turn only after
its predecessor in the tile's order started its release: the device-side
record that the reduction followed the schedule's order (DASH overview
(zskr.cn), section 2.1).
"""
import numpy as np
import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash
from deterministic_attention_backward_fa_gb300 import trace as T

from _gpu import Problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


# S, D, mask, schedule, dQ chains, split gangs, fill, CTA count (0 = the library's choice), timed ranks
TRACED = [(512, 128, False, "shift", 1, 0, 0, 0, 0), (512, 128, True, "symmetric_shift", 1, 0, 0, 0, 0),
          (1024, 64, True, "descending_q", 2, 0, 0, 0, 0), (512, 128, False, "atomic", 1, 0, 0, 0, 0),
          (1024, 128, False, "shift", 1, 2, 0, 8, 0), (1024, 64, True, "symmetric_shift", 2, 2, 0, 0, 0),
          (1024, 128, False, "shift", 1, 0, 1, 10, 0), (1024, 128, False, "shift", 1, 0, 0, 10, 1),
          (2048, 64, True, "symmetric_shift", 1, 0, 0, 11, 1)]


@pytest.mark.parametrize("S,D,causal,sched,chains,split,fill,ctas,timed", TRACED)
def test_trace_stamps_every_task_in_order(S, D, causal, sched, chains, split, fill, ctas, timed):
    P = Problem(1, 3, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    BH, n = 3, S // 128
    tasks, off, ctas = T.task_table(BH, n, causal, sched, sms, fill=bool(fill), chains=chains, split=split, ctas=ctas,
                                    timed=bool(timed))
    tr, _, _, same = T.run(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, tasks, off, 128, chains,
                           steps=1, warmup=1, split=split, ctas=ctas, fill=fill, rank_order=timed)
    if sched != "atomic":   # atomic adds land in no fixed order, so only the ordered schedules repeat bits
        assert same, "the traced kernel changed the results"
    assert (tr[:, [T.MMA_DP, T.MMA_DV, T.MMA_DQ, T.MMA_END, T.RED_Q, T.RED_LD, T.ACQ0, T.ACQ1, T.REL0,
                   T.REL1]] > 0).all(), "a task was not stamped"
    for a, b in ((T.MMA_DP, T.MMA_DV), (T.MMA_DV, T.MMA_DQ), (T.MMA_DQ, T.MMA_END), (T.PASS_A0, T.PASS_A1),
                 (T.PASS_A1, T.PASS_B0), (T.PASS_B0, T.PASS_B1), (T.RED_Q, T.RED_LD), (T.ACQ0, T.ACQ1),
                 (T.ACQ1, T.REL0), (T.REL0, T.REL1), (T.PASS_A1, T.PASS_A_LAST), (T.PASS_B1, T.PASS_B_LAST),
                 (T.PASS_A_LAST, T.MMA_DV)):
        assert (tr[:, b] >= tr[:, a]).all(), f"slot {b} stamped before slot {a}"
    ctas_seen = {int(x) & 0xFFFF for x in tr[:, T.META]}
    assert ctas_seen == {c for c in range(ctas) if off[c + 1] > off[c]}
    if sched != "atomic":
        _, _, viol, _ = T.summarize(tasks, off, tr, chains)
        assert viol == 0, f"{viol} ranks took their turn before their predecessor's release"
