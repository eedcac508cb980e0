"""Phase trace of the backward's main kernel (profiling).

Runs one workload's backward with the traced build of the main kernel
(dash_bwd_options_t.trace), which stamps every task's phases: the MMA warp's
issue points, the softmax passes, the dQ reduction's wait for the tile's turn
(DASH overview (zskr.cn), section 2.1: the serialised dQ reduction), its adds
and its release.  Prints a markdown summary: per-task phase durations, the
task period per CTA, and for an ordered schedule the hop of each dQ tile's
chain, from the release of one rank to the acquire of the next.

    python -m deterministic_attention_backward_fa_gb300.trace --workload full_s4096_d128 --schedule shift

The traced kernel returns the same bits as the plain one; its stamps cost a
few percent of throughput, which the summary reports (plain against traced
main-kernel time on the same task table).
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

import numpy as np
import torch

from . import (TRACE_SLOTS, attn_fwd, dash_attn_bwd_ex, dash_build_schedule, dash_build_schedule_ex,
               dash_build_shift_fill, dash_build_split_schedule, dash_choose_ctas, dash_choose_split,
               dash_choose_split_ctas, dash_sync_status)

# slot indices (include/dash.h)
MMA_DP, MMA_DV, MMA_DQ, MMA_END = 0, 1, 2, 3
PASS_A0, PASS_A1, PASS_B0, PASS_B1 = 4, 5, 6, 7
RED_Q, RED_LD, ACQ0, ACQ1, RED_ISSUED, REL0, CLK_AT_ACQ0, META, REL1 = 8, 9, 10, 11, 12, 13, 14, 15, 16
PASS_A_LAST, PASS_B_LAST, MMA_DV_OUT, MMA_DS_SEEN = 17, 18, 19, 20

L2_FLUSH_BYTES = 256 << 20


def task_table(BH, n, causal, schedule, sms, fill=False, chains=1, split=1, ctas=0, timed=False):
    """The table the library would build for this call (same generator and CTA choice; `ctas`, if set,
    is the CTA count asked for; `timed`: rank_order = 1)."""
    if split == -1:   # the library's choice of split and CTA count
        split, P, _ = dash_choose_split(BH, n, causal, schedule, sms, ctas)
        ctas = ctas or P
    if timed:
        if split > 1:
            P = ctas or dash_choose_split_ctas(BH, n, causal, schedule, split, sms)
        else:
            P = ctas or min(sms, BH * (n // 2 if schedule == "symmetric_shift" else n))
        tasks, off, _ = dash_build_schedule_ex(BH, n, causal, schedule, max(split, 1), 1, P)
        return tasks, off, P
    if split > 1:
        P = ctas or dash_choose_split_ctas(BH, n, causal, schedule, split, sms)
        tasks, off, _ = dash_build_split_schedule(BH, n, causal, schedule, split, P)
        return tasks, off, P
    if fill:
        tasks, off, P, _, _, _ = dash_build_shift_fill(BH, n, causal, schedule, ctas or sms)
        return tasks, off, P
    if ctas:
        P = ctas
    elif chains == 2 and schedule == "shift":
        P = min(sms, BH * n)
    else:
        P = dash_choose_ctas(BH, n, causal, schedule, sms)
    tasks, off, _ = dash_build_schedule(BH, n, causal, schedule, P)
    return tasks, off, P


def run(q, k, v, o, do, lse, causal, scale, schedule, tasks, off, tile=128, chains=1, steps=5, warmup=3,
        die_aware=0, cluster_size=0, supply_table=False, split=0, ctas=0, fill=0, rank_order=0):
    """Times the main kernel plain and traced on the same table; returns (trace int64 [n_tasks,
    TRACE_SLOTS] of the last traced run, plain ms, traced ms, outputs equal).  The kernel runs the
    library's own table, which task_table reproduces (with its cluster hand-offs, or die-aware
    placement); supply_table passes `tasks` instead (then without either)."""
    dev = q.device
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    tr = torch.zeros((len(tasks), TRACE_SLOTS), dtype=torch.int64, device=dev)
    outs = {}
    ms = {}
    for traced in (False, True):
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        times = []
        for i in range(warmup + steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)   # creates the events, whose handles the library records into
            b.record(stream)
            table = {"tasks": tasks, "cta_off": off} if supply_table else {}
            dash_attn_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, causal, scale, schedule, tile=tile,
                             main_events=(a, b), dq_chains=chains, trace=tr if traced else None,
                             die_aware=die_aware, cluster_size=cluster_size, shift_split=split, shift_fill=fill,
                             rank_order=rank_order,
                             num_ctas=0 if supply_table else ctas, **table)
            b.synchronize()
            if i >= warmup:
                times.append(a.elapsed_time(b))
        dash_sync_status()
        ms[traced] = statistics.median(times)
        outs[traced] = (dq, dk, dv)
    same = all(torch.equal(x, y) for x, y in zip(outs[False], outs[True]))
    return tr.cpu().numpy(), ms[False], ms[True], same


def _q(x):
    x = np.asarray(x, dtype=np.float64)
    if x.size == 0:
        return "—"
    p10, p50, p90 = np.percentile(x, [10, 50, 90])
    return f"{p50:,.0f} ({p10:,.0f} – {p90:,.0f})"


def summarize(tasks, off, tr, chains=1):
    """Phase statistics of one traced run, as markdown table rows (median, p10 – p90)."""
    tasks = np.asarray(tasks)
    P = len(off) - 1
    rows = []
    # SM clock from the (clk, ns) pairs of each CTA
    mhz = []
    for c in range(P):
        sl = slice(off[c], off[c + 1])
        ck, ns = tr[sl, CLK_AT_ACQ0].astype(np.float64), tr[sl, ACQ0].astype(np.float64)
        if len(ck) >= 2 and ns[-1] > ns[0]:
            mhz.append((ck[-1] - ck[0]) / (ns[-1] - ns[0]) * 1e3)
    sm_mhz = statistics.median(mhz) if mhz else float("nan")
    same_run = np.zeros(len(tasks), dtype=bool)     # task t+1 continues t's KV run on the same CTA
    for c in range(P):
        for t in range(off[c], off[c + 1] - 1):
            same_run[t] = not (tasks[t + 1, 3] & (1 << 28))
    nxt = np.nonzero(same_run)[0]
    d = lambda a, b, idx=slice(None): (tr[idx, b] - tr[idx, a]).astype(np.float64)
    rows.append(("task period on a CTA (dP^T issue to the next dP^T issue), clk",
                 _q(tr[nxt + 1, MMA_DP] - tr[nxt, MMA_DP])))
    rows.append(("MMA warp: dP^T issued until P is ready (pass A), clk", _q(d(MMA_DP, MMA_DV))))
    rows.append(("MMA warp: dV (+ next S^T) issued until dS is ready (pass B), clk", _q(d(MMA_DV, MMA_DQ))))
    rows.append(("  of which issuing dV (and the next S^T), clk", _q(d(MMA_DV, MMA_DV_OUT))))
    rows.append(("  of which waiting for dS, clk", _q(d(MMA_DV_OUT, MMA_DS_SEEN))))
    rows.append(("MMA warp: dQ and dK issued, clk", _q(d(MMA_DQ, MMA_END))))
    rows.append(("MMA warp: end of task until the next dP^T (Q/dO landed, dQ drained), clk",
                 _q(tr[nxt + 1, MMA_DP] - tr[nxt, MMA_END])))
    rows.append(("pass A (S^T -> P), clk", _q(d(PASS_A0, PASS_A1))))
    rows.append(("pass A end until pass B starts (dP^T landed, dS buffer free), clk", _q(d(PASS_A1, PASS_B0))))
    rows.append(("pass B (dP^T -> dS), clk", _q(d(PASS_B0, PASS_B1))))
    rows.append(("pass A: softmax warp 4 done until the last softmax warp is done, clk", _q(d(PASS_A1, PASS_A_LAST))))
    rows.append(("pass B: softmax warp 4 done until the last softmax warp is done, clk", _q(d(PASS_B1, PASS_B_LAST))))
    rows.append(("pass B end until the next pass A starts (next S^T done, its LSE landed), clk",
                 _q(tr[nxt + 1, PASS_A0] - tr[nxt, PASS_B1])))
    rows.append(("dQ MMA issued until the partial is in registers, clk", _q(d(MMA_DQ, RED_LD))))
    rows.append(("reduction warps: wait for the tile's turn, ns", _q(d(ACQ0, ACQ1))))
    rows.append(("reduction warps: turn taken until every add is issued, ns", _q(d(ACQ1, REL0))))
    rows.append(("release store (its fence waits for the adds), ns", _q(d(REL0, REL1))))
    # hops of the ordered dQ chains
    rank = tasks[:, 3] & ((1 << 24) - 1)
    hop0, hop1, viol = [], [], 0
    if chains >= 1:   # chains = 0: the atomic schedule, whose adds have no order
        key = {}
        for t in range(len(tasks)):
            bh, _, qq = int(tasks[t, 0]), int(tasks[t, 1]), int(tasks[t, 2])
            r = int(rank[t])
            key[(bh, qq, r % chains, r // chains)] = t
        for (bh, qq, ch, pos), t in key.items():
            prev = key.get((bh, qq, ch, pos - 1))
            if prev is None:
                continue
            hop0.append(tr[t, ACQ1] - tr[prev, REL0])
            hop1.append(tr[t, ACQ1] - tr[prev, REL1])
            viol += int(tr[t, ACQ1] < tr[prev, REL0])
    rows.append(("hop: predecessor's release starts until this rank's turn is taken, ns", _q(hop0)))
    rows.append(("hop: predecessor's release returned until this rank's turn is taken, ns", _q(hop1)))
    smids = sorted({int(x) >> 16 for x in tr[:, META]})
    return rows, sm_mhz, viol, len(smids)


def main(argv=None):
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if here not in sys.path:
        sys.path.insert(0, here)
    import workloads
    from . import _build, lib
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="full_s4096_d128", choices=list(workloads.WORKLOADS))
    ap.add_argument("--schedule", default="shift")
    ap.add_argument("--fill", action="store_true")
    ap.add_argument("--chains", type=int, default=1)
    ap.add_argument("--die-aware", action="store_true", help="die-aware placement (shift schedules)")
    ap.add_argument("--cluster-size", type=int, default=0,
                    help="thread-block clusters of the dQ hand-offs: 0 or 1 = none, else the size")
    ap.add_argument("--split", type=int, default=0,
                    help="split gangs of shift and symmetric shift (shift_split; -1 = the library's choice)")
    ap.add_argument("--ctas", type=int, default=0, help="CTA count (num_ctas); 0 = the library's choice")
    ap.add_argument("--timed", action="store_true", help="timed ranks (rank_order = 1)")
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--out", default="")
    args = ap.parse_args(argv)
    if not _build.up_to_date():
        _build.build()
    lib()
    w = workloads.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in workloads.make_workload_inputs(w))
    o, lse = attn_fwd(q, k, v, w.causal, w.scale)
    dash_sync_status()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    BH, n = w.B * w.H, w.n_blocks
    tasks, off, P = task_table(BH, n, w.causal, args.schedule, sms, args.fill, args.chains, args.split, args.ctas,
                               args.timed)
    tr, plain_ms, traced_ms, same = run(q, k, v, o, do, lse, w.causal, w.scale, args.schedule, tasks, off,
                                        w.tile, args.chains, args.steps, die_aware=int(args.die_aware),
                                        cluster_size=args.cluster_size, split=args.split, ctas=args.ctas,
                                        fill=int(args.fill), rank_order=int(args.timed))
    rows, sm_mhz, viol, n_sms = summarize(tasks, off, tr, args.chains if args.schedule != "atomic" else 0)
    name = args.schedule + (" with fill" if args.fill else "") + (" two dQ chains" if args.chains == 2 else "")
    name += " die-aware" if args.die_aware else ""
    name += f", clusters of {args.cluster_size}" if args.cluster_size > 1 else ""
    name += (f", split gangs of {args.split}" if args.split > 1 else
             ", split gangs as the library picks them" if args.split == -1 else "")
    name += ", timed ranks" if args.timed else ""
    cmd = " ".join(["python -m deterministic_attention_backward_fa_gb300.trace"] + (argv or sys.argv[1:]))
    lines = [f"# Phase trace of dash_bwd_main: {w.name}, {name}", "",
             f"Command: `{cmd}`", "",
             f"- {w.describe()}; {len(tasks)} tasks on {P} CTAs ({n_sms} distinct SMs).",
             f"- main kernel {plain_ms:.3f} ms plain, {traced_ms:.3f} ms traced (same table), "
             f"{w.flops() / (plain_ms / 1e3) / 1e12:.0f} TFLOPS plain; traced outputs equal the plain ones "
             f"bit for bit: {same}.",
             f"- SM clock from the stamps: {sm_mhz:.0f} MHz. Five 128-row MMAs of one task take "
             f"5 x 8 x 64 = 2,560 clk of tensor-pipe time at D = 128 (1,280 at D = 64).",
             f"- ordered-chain violations (a rank's turn taken before its predecessor's release began): {viol}.",
             "", "| phase (per task) | median (p10 – p90) |", "|---|---:|"]
    lines += [f"| {a} | {b} |" for a, b in rows]
    text = "\n".join(lines) + "\n"
    print(text)
    if args.out:
        with open(args.out, "w") as fh:
            fh.write(text)
    return 0


if __name__ == "__main__":
    sys.exit(main())
