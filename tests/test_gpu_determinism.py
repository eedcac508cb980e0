"""Run-to-run bit identity of the deterministic schedules, and the bounded
device waits.

Every schedule except atomic must give bit-identical dQ, dK, dV and fp32 dQ
accumulator across 100 runs on each of the five named workloads.  The timeout
test hands the kernel a task table whose dQ reduction order skips a rank, so
that a semaphore wait can never succeed; the wait must run out after its limit
and the status must say so, with the CUDA context still usable afterwards.
"""
import numpy as np
import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash
import workloads

from _gpu import Problem, assert_close

pytestmark = pytest.mark.gpu

RUNS = 100


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


WL = list(workloads.WORKLOADS.values())


@pytest.mark.parametrize("w", WL, ids=[w.name for w in WL])
def test_bit_identical_across_runs(w):
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    atomic_identical = None
    for sched in w.schedules:
        first = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, dq_accum=True, tile=w.tile)
        same = True
        outs = [torch.empty_like(x) for x in first]
        for _ in range(RUNS - 1):
            dash.dash_attn_bwd_ex(P.q, P.k, P.v, o, P.do, lse, outs[0], outs[1], outs[2], w.causal, P.scale,
                                  sched, tile=w.tile, dq_accum_out=outs[3])
            same = same and all(torch.equal(a, b) for a, b in zip(outs, first))
        dash.dash_sync_status()
        if sched == "atomic":
            atomic_identical = same
        else:
            assert same, f"{w.name}: schedule {sched} is not bit-identical across {RUNS} runs"
    print(f"{w.name}: atomic bit-identical across {RUNS} runs: {atomic_identical}")


@pytest.mark.parametrize("wname", ["full_s4096_d128", "causal_s16384_d128"])
def test_two_dq_chains_bit_identical_across_runs(wname):
    # the two-chain reduction is deterministic too: its order is fixed by rank parity
    w = workloads.WORKLOADS[wname]
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    for sched in w.schedules:
        if sched == "atomic":
            continue
        first = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, dq_accum=True, tile=w.tile,
                              dq_chains=2)
        outs = [torch.empty_like(x) for x in first]
        same = True
        for _ in range(RUNS - 1):
            dash.dash_attn_bwd_ex(P.q, P.k, P.v, o, P.do, lse, outs[0], outs[1], outs[2], w.causal, P.scale,
                                  sched, tile=w.tile, dq_accum_out=outs[3], dq_chains=2)
            same = same and all(torch.equal(a, b) for a, b in zip(outs, first))
        dash.dash_sync_status()
        assert same, f"{wname}: {sched} with two dQ chains is not bit-identical across {RUNS} runs"
        # dK and dV do not depend on the dQ order; dQ is within rounding of the one-chain order
        one = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, tile=w.tile)
        assert torch.equal(one[1], first[1]) and torch.equal(one[2], first[2])
        assert_close(f"{sched} two vs one chain dQ", first[0].float(), one[0].double().cpu().numpy(),
                     rel=2e-3, abs_=1e-2)


SPLIT_WL = [w for w in WL if w.S >= 4096]


@pytest.mark.parametrize("w", SPLIT_WL, ids=[w.name for w in SPLIT_WL])
def test_split_gangs_bit_identical_across_runs(w):
    # split gangs as the library picks them (an extension): a fixed (sub-gang, step) order per tile
    sched = "symmetric_shift" if w.causal else "shift"
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    first = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, dq_accum=True, tile=w.tile,
                          shift_split=-1)
    outs = [torch.empty_like(x) for x in first]
    same = True
    for _ in range(RUNS - 1):
        dash.dash_attn_bwd_ex(P.q, P.k, P.v, o, P.do, lse, outs[0], outs[1], outs[2], w.causal, P.scale,
                              sched, tile=w.tile, dq_accum_out=outs[3], shift_split=-1)
        same = same and all(torch.equal(a, b) for a, b in zip(outs, first))
    dash.dash_sync_status()
    assert same, f"{w.name}: {sched} with split gangs is not bit-identical across {RUNS} runs"
    # dK and dV do not depend on the dQ order
    one = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, tile=w.tile)
    assert torch.equal(one[1], first[1]) and torch.equal(one[2], first[2])


@pytest.mark.parametrize("wname,sched", [("causal_s16384_d128", "symmetric_shift"), ("full_s4096_d128", "shift"),
                                         ("causal_s8192_d64", "symmetric_shift")])
def test_timed_ranks_bit_identical_across_runs(wname, sched):
    # timed ranks (an extension) on every SM: the order comes from a deterministic simulation, so the bits repeat
    w = workloads.WORKLOADS[wname]
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    first = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, dq_accum=True, tile=w.tile,
                          rank_order=1)
    outs = [torch.empty_like(x) for x in first]
    same = True
    for _ in range(RUNS - 1):
        dash.dash_attn_bwd_ex(P.q, P.k, P.v, o, P.do, lse, outs[0], outs[1], outs[2], w.causal, P.scale,
                              sched, tile=w.tile, dq_accum_out=outs[3], rank_order=1)
        same = same and all(torch.equal(a, b) for a, b in zip(outs, first))
    dash.dash_sync_status()
    assert same, f"{wname}: {sched} with timed ranks is not bit-identical across {RUNS} runs"


def test_deterministic_schedules_agree_within_tolerance():
    # different schedules reduce dQ in different orders: close, not equal bits
    w = workloads.WORKLOADS["causal_s2048_d128"]
    P = Problem(2, 4, 1024, 128, True)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, True, P.scale)
    ref = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "serial")
    for sched in ("descending_q", "symmetric_shift", "atomic"):
        got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, sched)
        for a, b in zip(got, ref):
            assert_close(sched, a.float(), b.double().cpu().numpy(), rel=2e-3, abs_=1e-2)
        if sched == "atomic":
            # same chains as serial, so dK/dV accumulate in the same order; only dQ's order differs
            assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    assert w.causal


def test_stuck_semaphore_times_out_and_context_survives():
    P = Problem(1, 2, 512, 128, False)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, False, P.scale)
    ref = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, False, P.scale, "serial")
    tasks, off, _ = dash.dash_build_schedule(2, 4, False, "serial", 4)
    tasks = tasks.copy()
    # give a rank-1 task rank 2: its tile's order now skips rank 1
    i = int(np.nonzero((tasks[:, 3] & dash.TASK_RANK_MASK) == 1)[0][0])
    tasks[i, 3] = (tasks[i, 3] & ~dash.TASK_RANK_MASK) | 2
    dq, dk, dv = (torch.empty_like(P.q) for _ in range(3))
    # the host check refuses such a table before the launch ...
    with pytest.raises(dash.DashError) as ei:
        dash.dash_attn_bwd_ex(P.q, P.k, P.v, o, P.do, lse, dq, dk, dv, False, P.scale, "serial",
                              tasks=tasks, cta_off=off, spin_limit_ns=50_000_000)
    assert ei.value.code == 6, str(ei.value)
    # ... and, told to trust it, the device's bounded waits run out and say so
    dash.dash_attn_bwd_ex(P.q, P.k, P.v, o, P.do, lse, dq, dk, dv, False, P.scale, "serial",
                          tasks=tasks, cta_off=off, spin_limit_ns=50_000_000, trust_table=1)
    with pytest.raises(dash.DashError) as ei:
        dash.dash_sync_status()
    assert ei.value.code == 4, str(ei.value)
    dash.dash_sync_status()   # the status word was cleared
    again = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, False, P.scale, "serial")
    dash.dash_sync_status()
    for a, b in zip(again, ref):
        assert torch.equal(a, b)


def test_supplied_table_equal_to_generated_gives_same_bits():
    P = Problem(1, 2, 512, 128, True)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, True, P.scale)
    ref = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "symmetric_shift", num_ctas=4)
    tasks, off, _ = dash.dash_build_schedule(2, 4, True, "symmetric_shift", 4)
    got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, True, P.scale, "symmetric_shift", tasks=tasks, cta_off=off)
    dash.dash_sync_status()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("wname,sched", [("full_s4096_d128", "shift"), ("causal_s8192_d64", "symmetric_shift")])
def test_fill_bit_identical_across_runs(wname, sched):
    # fill (an extension): each head's order is its own schedule's
    w = workloads.WORKLOADS[wname]
    P = Problem(w.B, w.H, w.S, w.D, w.causal, w.gain)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, w.causal, P.scale)
    first = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, w.causal, P.scale, sched, dq_accum=True, tile=w.tile,
                          shift_fill=1)
    outs = [torch.empty_like(x) for x in first]
    same = True
    for _ in range(RUNS - 1):
        dash.dash_attn_bwd_ex(P.q, P.k, P.v, o, P.do, lse, outs[0], outs[1], outs[2], w.causal, P.scale, sched,
                              tile=w.tile, dq_accum_out=outs[3], shift_fill=1)
        same = same and all(torch.equal(a, b) for a, b in zip(outs, first))
    dash.dash_sync_status()
    assert same, f"{wname}: {sched} with fill is not bit-identical across {RUNS} runs"


@pytest.mark.parametrize("causal,sched", [(False, "shift"), (False, "serial"), (True, "symmetric_shift"),
                                          (True, "descending_q")])
def test_same_bits_whatever_the_cta_count(causal, sched):
    # a dQ tile's rank order is fixed by the schedule (KV index or step), not by
    # which CTA runs which chain, so every CTA count gives the same bits
    P = Problem(2, 3, 1024, 128, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    ref = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched)
    gang = 8 if sched == "shift" else 4 if sched == "symmetric_shift" else 1
    for ctas in (gang, 3 * gang, 6 * gang):
        got = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched, num_ctas=ctas)
        dash.dash_sync_status()
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.equal(a, b), f"{sched} on {ctas} CTAs: {name} differs"
