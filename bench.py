#!/usr/bin/env python
"""Throughput of the deterministic attention backward on GB300.

One step = one dash_attn_bwd call (preprocess, persistent main kernel, dQ
convert) over the whole workload, inputs resident in HBM, L2 flushed between
steps.  Every schedule valid for the workload is timed; `value` is the best
deterministic schedule's TFLOPS (conventional count: 10*B*H*S^2*D for a full
mask, half of it for a causal one) and the atomic schedule gives the ratio.
The ordered schedules are timed a second time with the optional two-chain dQ
reduction (dq_chains = 2, a different fixed summation order); those figures go
to `extension_two_dq_chains` and never into `value`.  Shift and symmetric shift
are also timed with fill (shift_fill = 1: the SMs that whole gangs of their
chains leave idle run some heads in the serial or descending order), under
`extension_fill`, never in `value`; and with die-aware placement (die_aware = 1:
each gang of chains on one die, its semaphores homed there) under
`extension_die_aware`, and with split gangs (shift_split = -1: each head's gang
runs as k sub-gangs, k picked by the library's simulation, so that the CTA
count need only be a multiple of a sub-gang) under `extension_split`, and with
timed ranks (rank_order = 1: each dQ tile reduced in the order the scheduled
chains reach it, on every SM) under `extension_timed`, never in `value`.  The long causal workload
(causal_s16384_d128) is timed in the same run, every schedule of its mask and
symmetric shift with fill, die-aware placement and split gangs, and reported
under `workloads` with its own ratio
to atomic and roofline fraction (`--also` names other workloads; '' skips it).

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

--sweep times the pages' sweep instead (16384 tokens, S = 512 ... 16384, D = 64
and 128, both masks) and prints one JSON line per configuration.

--impl reference times the fp64 CPU oracle on the host cores instead (one head
of the workload per step).  Under torchrun each rank runs an independent
replica of the workload on its own GPU (there is no data exchange); rank 0
prints the JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "deterministic attn-bwd TFLOPS & % BF16 peak; ratio vs own atomicAdd bwd"
DEFAULT_WORKLOAD = "full_s4096_d128"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = ["bwd.cu", "sm103.cuh", "kernels.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--schedules", default="", help="comma-separated subset of the workload's schedules")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-two-chains", action="store_true",
                    help="skip timing the optional two-chain dQ reduction (dq_chains = 2)")
    ap.add_argument("--no-shift-fill", action="store_true",
                    help="skip timing shift and symmetric shift with fill (shift_fill = 1)")
    ap.add_argument("--no-die-aware", action="store_true",
                    help="skip timing shift and symmetric shift with die-aware placement (die_aware = 1)")
    ap.add_argument("--split", type=int, default=-1,
                    help="split gangs timed for shift and symmetric shift (shift_split: -1 = the library's "
                         "choice, k > 1 = k sub-gangs, 0 or 1 skips)")
    ap.add_argument("--no-timed", action="store_true",
                    help="skip timing shift and symmetric shift with timed ranks (rank_order = 1)")
    ap.add_argument("--also", default="causal_s16384_d128",
                    help="comma-separated further workloads timed in the same run and reported under "
                         "`workloads` (every schedule of the mask and fill; '' for none)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the pages' sweep (16384 tokens, S = 512..16384, D = 64/128, both masks) "
                         "and print one JSON line per configuration instead of the bench line")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, total_s: float) -> float:
    """Throughput of the whole job: every rank runs its own replica of the workload."""
    return world * flops_per_step * steps / total_s / 1e12


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "deterministic_attention_backward_fa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return {"bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in (self.out or "").splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(w, seconds: float):
    """The fp64 oracle's backward, head by head, until `seconds` have passed."""
    from oracle import attention as A
    q, k, v, do = (t.double().numpy() for t in workloads.make_workload_inputs(w))
    flops_head = w.flops() / (w.B * w.H)
    done, spent = 0, 0.0
    for b in range(w.B):
        for h in range(w.H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            o, lse = A.forward(q[sl], k[sl], v[sl], w.causal, w.scale)
            t0 = time.perf_counter()
            A.backward(q[sl], k[sl], v[sl], o, do[sl], lse, w.causal, w.scale)
            spent += time.perf_counter() - t0
            done += 1
            if spent >= seconds:
                break
        if spent >= seconds:
            break
    return {"value": done * flops_head / spent / 1e12, "unit": "TFLOPS", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle backward on {done} of {w.B * w.H} heads of {w.name} "
                      f"({spent:.1f} s), O/LSE from the oracle forward outside the timing"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = workloads.WORKLOADS[args.workload]
    from oracle import attention as A
    q, k, v, do = (t.double().numpy() for t in workloads.make_workload_inputs(w))
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    pre = {}
    for i in range(args.warmup + args.steps):
        b, h = heads[i % len(heads)]
        if (b, h) not in pre:
            sl = (slice(b, b + 1), slice(h, h + 1))
            pre[(b, h)] = A.forward(q[sl], k[sl], v[sl], w.causal, w.scale)
    times = []
    for i in range(args.warmup + args.steps):
        b, h = heads[i % len(heads)]
        sl = (slice(b, b + 1), slice(h, h + 1))
        o, lse = pre[(b, h)]
        t0 = time.perf_counter()
        A.backward(q[sl], k[sl], v[sl], o, do[sl], lse, w.causal, w.scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    flops_head = w.flops() / (w.B * w.H)
    total = sum(times)
    value = len(times) * flops_head / total / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                       "mask": "causal" if w.causal else "full", "step": "oracle backward of one head"},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"one head of {w.name} per step, fp64 numpy"},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def split_of(w, sched, k):
    """The shift_split to time for the schedule on this workload: -1 (the library's choice) or k where k
    divides its gang; 0 where split gangs do not apply."""
    if k in (0, 1) or sched not in ("shift", "symmetric_shift") or sched not in w.schedules:
        return 0
    if k == -1:
        return -1
    n = w.S // w.tile
    gang = n // 2 if sched == "symmetric_shift" else n
    return k if k > 1 and gang % k == 0 else 0


def split_chosen(dash, w, sched, k, sms):
    """The split a run with shift_split = k uses (-1 resolved through the library's choice)."""
    return dash.dash_choose_split(w.B * w.H, w.S // w.tile, w.causal, sched, sms)[0] if k == -1 else k


def best_with_extensions(results, two_chains, fill, best, world, peak, die=None, split=None, timed=None):
    """The fastest deterministic layout including the extensions (never in `value`)."""
    cands = {best: results[best]}
    cands.update({f"{s}+split": r for s, r in (split or {}).items()})
    cands.update({f"{s}+timed": r for s, r in (timed or {}).items()})
    cands.update({f"{s}+fill": r for s, r in fill.items()})
    cands.update({f"{s}+two_dq_chains": r for s, r in two_chains.items()})
    cands.update({f"{s}+die_aware": r for s, r in (die or {}).items()})
    name = max(cands, key=lambda s: cands[s]["tflops"])
    r = cands[name]
    return {"schedule": name, "tflops": r["tflops"], "ratio_vs_atomic": r.get("vs_atomic"),
            "pct_bf16_peak": 100.0 * r["tflops"] / world / peak}


def runtime_choice(dash, w, sms, atomic_ms, serial_ms, measured_best, measured_best_split=None,
                   measured_best_layout=None):
    """The library's runtime schedule choice with task costs fitted to this run's atomic and
    serial times, against the schedule measured best; with `measured_best_split` (the best of the
    pages' schedules and split gangs, e.g. "shift+split"), also the split-aware choice against it; with
    `measured_best_layout` (the best of those and timed ranks), also dash_choose_layout against it."""
    BH, n = w.B * w.H, w.S // w.tile
    c, r = dash.dash_fit_costs(BH, n, w.causal, sms, atomic_ms, serial_ms)
    chosen, ctas, _ = dash.dash_choose_schedule(BH, n, w.causal, sms, c, r)
    out = {"cost_c": c, "cost_r": r, "chosen": chosen, "ctas": ctas, "measured_best": measured_best,
           "agrees": chosen == measured_best}
    if measured_best_split is not None:
        name, ctas_s, k, _ = dash.dash_choose_schedule_split(BH, n, w.causal, sms, c, r)
        label = f"{name}+split" if k > 1 else name
        out["with_split"] = {"chosen": label, "split": k, "ctas": ctas_s, "measured_best": measured_best_split,
                             "agrees": label == measured_best_split}
    if measured_best_layout is not None:
        name, ctas_l, k, ro, _ = dash.dash_choose_layout(BH, n, w.causal, sms, c, r)
        label = name + ("+split" if k > 1 else "") + ("+timed" if ro else "")
        out["layout"] = {"chosen": label, "split": k, "rank_order": ro, "ctas": ctas_l,
                         "measured_best": measured_best_layout, "agrees": label == measured_best_layout}
    return out


def best_label(det, split, timed=None):
    """The fastest of the pages' schedules (TFLOPS by name), the split-gang runs and the timed-rank runs, split
    gangs labelled "<schedule>+split" where they were timed with a split above one, timed ranks "<schedule>+timed"."""
    cands = dict(det)
    for s_, (t, k) in split.items():
        if k > 1:
            cands[f"{s_}+split"] = t
    for s_, t in (timed or {}).items():
        cands[f"{s_}+timed"] = t
    return max(cands, key=cands.get)


def run_sweep(args, dash):
    """The pages' sweep, one GPU: every configuration and every schedule valid for its mask,
    timed like the bench line (event-timed steps, L2 flushed between steps)."""
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    peaks, _ = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    for w in workloads.pages_sweep():
        q, k_, v, do = (t.to(dev) for t in workloads.make_workload_inputs(w))
        o, lse = dash.attn_fwd(q, k_, v, w.causal, w.scale)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        res, fill, split, timed = {}, {}, {}, {}
        runs = [(s, 0, 0, 0) for s in w.schedules]
        runs += [(s, 1, 0, 0) for s in ("shift", "symmetric_shift") if s in w.schedules and not args.no_shift_fill]
        runs += [(s, 0, split_of(w, s, args.split), 0) for s in ("shift", "symmetric_shift")
                 if split_of(w, s, args.split)]
        runs += [(s, 0, 0, 1) for s in ("shift", "symmetric_shift") if s in w.schedules and not args.no_timed]
        with ClockSampler(0) as clk:
            for sched, shift_fill, k, ro in runs:
                for _ in range(args.warmup):
                    flush.fill_(1)
                    dash.dash_attn_bwd_ex(q, k_, v, o, do, lse, dq, dk, dv, w.causal, w.scale, sched, tile=w.tile,
                                          shift_fill=shift_fill, shift_split=k, rank_order=ro)
                dash.dash_sync_status()
                ms = []
                for _ in range(args.steps):
                    flush.fill_(1)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    dash.dash_attn_bwd_ex(q, k_, v, o, do, lse, dq, dk, dv, w.causal, w.scale, sched, tile=w.tile,
                                          shift_fill=shift_fill, shift_split=k, rank_order=ro)
                    b.record(stream)
                    b.synchronize()
                    ms.append(a.elapsed_time(b))
                dash.dash_sync_status()
                tf = w.flops() / (statistics.median(ms) / 1e3) / 1e12
                (timed if ro else split if k else fill if shift_fill else res)[sched] = tf
        det = {s: t for s, t in res.items() if s != "atomic"}
        best = max(det, key=det.get)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        ks = {s_: split_chosen(dash, w, s_, args.split, sms) for s_ in split}
        choice = runtime_choice(dash, w, sms, 1.0 / res["atomic"], 1.0 / res["serial"], best,
                                best_label(det, {s_: (t, ks[s_]) for s_, t in split.items()}),
                                best_label(det, {s_: (t, ks[s_]) for s_, t in split.items()}, timed))
        print(json.dumps({"sweep": "pages_16k_tokens", "workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                          "mask": "causal" if w.causal else "full", "tile": w.tile, "unit": "TFLOPS",
                          "statistic": f"median of {args.steps} steps", "schedules": res,
                          "best_deterministic": best, "pct_bf16_peak": 100.0 * det[best] / peak,
                          "ratio_vs_atomic": det[best] / res["atomic"], "extension_fill": fill or None,
                          "extension_split": {s: {"tflops": t, "vs_atomic": t / res["atomic"], "split": ks[s]}
                                              for s, t in split.items()} or None,
                          "extension_timed": {s: {"tflops": t, "vs_atomic": t / res["atomic"]}
                                              for s, t in timed.items()} or None,
                          "runtime_choice": choice, "clocks": clk.summary()}), flush=True)
        del q, k_, v, do, o, lse, dq, dk, dv
        torch.cuda.empty_cache()


def time_runs(dash, w, tensors, runs, args, flush, stream, world, dev, barrier):
    """Times each (schedule, dq_chains, shift_fill, die_aware, shift_split, rank_order) of `runs`: W warm-up steps,
    then K steps, each
    bracketed by CUDA events on the launching stream, with the main kernel's own events inside."""
    q, k, v, o, do, lse, dq, dk, dv = tensors
    flops = w.flops()
    results, two_chains, fill, die, split, timed = {}, {}, {}, {}, {}, {}
    launches = 0
    for sched, chains, shift_fill, die_aware, ks, ro in runs:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for e in evs:
            for x in e:
                x.record(stream)
        for _ in range(args.warmup):
            flush.fill_(1)
            dash.dash_attn_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, sched, tile=w.tile,
                                  dq_chains=chains, shift_fill=shift_fill, die_aware=die_aware, shift_split=ks,
                                  rank_order=ro)
        dash.dash_sync_status()
        barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(1)   # evict the previous step's working set from L2
            evs[i][0].record(stream)
            dash.dash_attn_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale, sched, tile=w.tile,
                                  main_events=(evs[i][1], evs[i][2]), dq_chains=chains,
                                  shift_fill=shift_fill, die_aware=die_aware, shift_split=ks, rank_order=ro)
            evs[i][3].record(stream)
        torch.cuda.synchronize()
        barrier()
        dash.dash_sync_status()
        launches += dash.KERNELS_PER_BWD * args.steps
        step_ms = [evs[i][0].elapsed_time(evs[i][3]) for i in range(args.steps)]
        main_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(args.steps)]
        total_s = max_over_ranks(sum(step_ms) / 1e3, world, dev)
        out = (timed if ro else split if ks else die if die_aware else fill if shift_fill else
               results if chains == 1 else two_chains)
        out[sched] = {"ms": 1e3 * total_s / args.steps, "main_ms": statistics.mean(main_ms),
                      "tflops": whole_job_tflops(world, flops, args.steps, total_s)}
        if ks:
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            out[sched]["split"] = split_chosen(dash, w, sched, ks, sms)
    return results, two_chains, fill, die, split, timed, launches


def time_other_workload(dash, w, args, flush, stream, world, dev, barrier):
    """Every schedule of the workload's mask (one dQ chain) and shift / symmetric shift with fill, timed
    like the main line; summarised with the best of the pages' deterministic schedules, its ratio to
    atomic and the main kernel's roofline fraction."""
    q, k, v, do = (t.to(dev) for t in workloads.make_workload_inputs(w))
    o, lse = dash.attn_fwd(q, k, v, w.causal, w.scale)
    dash.dash_sync_status()
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    runs = [(s, 1, 0, 0, 0, 0) for s in w.schedules]
    runs += [(s, 1, 1, 0, 0, 0) for s in ("shift", "symmetric_shift") if s in w.schedules and not args.no_shift_fill]
    runs += [(s, 1, 0, 1, 0, 0) for s in ("shift", "symmetric_shift") if s in w.schedules and not args.no_die_aware]
    runs += [(s, 1, 0, 0, split_of(w, s, args.split), 0) for s in ("shift", "symmetric_shift")
             if split_of(w, s, args.split)]
    runs += [(s, 1, 0, 0, 0, 1) for s in ("shift", "symmetric_shift") if s in w.schedules and not args.no_timed]
    tensors = (q, k, v, o, do, lse, dq, dk, dv)
    results, _, fill, die, split, timed, launches = time_runs(dash, w, tensors, runs, args, flush, stream, world, dev,
                                                              barrier)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    atomic = results["atomic"]
    for r in (list(results.values()) + list(fill.values()) + list(die.values()) + list(split.values())
              + list(timed.values())):
        r["vs_atomic"] = r["tflops"] / atomic["tflops"]
    det = {s: r for s, r in results.items() if s != "atomic"}
    best = max(det, key=lambda s: det[s]["tflops"])
    achieved = w.flops() / (results[best]["main_ms"] / 1e3) / 1e12
    out = {"config": {"B": w.B, "H": w.H, "S": w.S, "D": w.D, "mask": "causal" if w.causal else "full",
                      "tile": w.tile, "flops_per_step": w.flops()},
           "best_deterministic": best, "tflops": results[best]["tflops"],
           "pct_bf16_peak": 100.0 * results[best]["tflops"] / world / peak,
           "ratio_vs_atomic": results[best]["vs_atomic"], "schedules": results,
           "extension_fill": fill or None,
           "extension_die_aware": die or None,
           "extension_split": split or None,
           "extension_timed": timed or None,
           "best_with_extensions": best_with_extensions(results, {}, fill, best, world, peak, die, split, timed),
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                        "frac": achieved / peak, "kernel": "dash_bwd_main",
                        "peak_source": f"{peak_kind} bf16_tflops (burst)"},
           "launches": launches}
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    return out



def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.sweep:
        import deterministic_attention_backward_fa_gb300 as dash
        from deterministic_attention_backward_fa_gb300 import _build
        torch.cuda.set_device(0)
        if not _build.up_to_date():
            _build.build()
        dash.lib()
        return run_sweep(args, dash)

    import deterministic_attention_backward_fa_gb300 as dash
    from deterministic_attention_backward_fa_gb300 import _build

    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0 or not _build.up_to_date():
        _build.build()
    if world > 1:
        dist.barrier()
    dash.lib()

    w = workloads.WORKLOADS[args.workload]
    dev = torch.device("cuda", local_rank)
    host = workloads.make_workload_inputs(w)
    q, k, v, do = (t.to(dev) for t in host)
    o, lse = dash.attn_fwd(q, k, v, w.causal, w.scale)
    dash.dash_sync_status()
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    flops = w.flops()

    def barrier():
        if world > 1:
            torch.distributed.barrier()


    gpu_index = local_rank
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local_rank])
        except (ValueError, IndexError):
            pass

    scheds = [s for s in w.schedules if not args.schedules or s in args.schedules.split(",")]
    runs = [(s, 1, 0, 0, 0, 0) for s in scheds]
    runs += [(s, 2, 0, 0, 0, 0) for s in scheds if s != "atomic" and not args.no_two_chains]
    runs += [(s, 1, 1, 0, 0, 0) for s in ("shift", "symmetric_shift") if s in scheds and not args.no_shift_fill]
    runs += [(s, 1, 0, 1, 0, 0) for s in ("shift", "symmetric_shift") if s in scheds and not args.no_die_aware]
    runs += [(s, 1, 0, 0, split_of(w, s, args.split), 0) for s in ("shift", "symmetric_shift")
             if s in scheds and split_of(w, s, args.split)]
    runs += [(s, 1, 0, 0, 0, 1) for s in ("shift", "symmetric_shift") if s in scheds and not args.no_timed]
    with ClockSampler(gpu_index) as clk:
        tensors = (q, k, v, o, do, lse, dq, dk, dv)
        results, two_chains, fill, die, split, timed, launches = time_runs(dash, w, tensors, runs, args, flush, stream,
                                                                           world, dev, barrier)
        also = {}
        for name in [x for x in args.also.split(",") if x and x != w.name]:
            also[name] = time_other_workload(dash, workloads.WORKLOADS[name], args, flush, stream, world, dev,
                                             barrier)
            launches += also[name].pop("launches")
    clocks = clk.summary()

    det = {s: r for s, r in results.items() if s != "atomic"} or results
    best = max(det, key=lambda s: det[s]["tflops"])
    atomic = results.get("atomic")
    for s, r in (list(results.items()) + list(two_chains.items()) + list(fill.items()) + list(die.items())
                 + list(split.items()) + list(timed.items())):
        r["vs_atomic"] = r["tflops"] / atomic["tflops"] if atomic else None
    choice = None
    if atomic and "serial" in results:
        choice = runtime_choice(dash, w, torch.cuda.get_device_properties(dev).multi_processor_count,
                                atomic["main_ms"], results["serial"]["main_ms"], best,
                                best_label({s_: r["tflops"] for s_, r in det.items()},
                                           {s_: (r["tflops"], r["split"]) for s_, r in split.items()}),
                                best_label({s_: r["tflops"] for s_, r in det.items()},
                                           {s_: (r["tflops"], r["split"]) for s_, r in split.items()},
                                           {s_: r["tflops"] for s_, r in timed.items()}))

    # end to end through the host-buffer entry point: H2D inputs, backward, D2H gradients
    pin = [t.pin_memory() for t in host] + [o.cpu().pin_memory(), lse.cpu().pin_memory()]
    hq, hk, hv, hdo, ho, hl = pin
    outs = [torch.empty_like(hq).pin_memory() for _ in range(3)]
    for _ in range(0 if args.no_e2e else max(1, args.warmup)):
        dash.dash_attn_bwd_host(hq, hk, hv, ho, hdo, hl, *outs, w.causal, w.scale, best)
    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, 20))
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        dash.dash_attn_bwd_host(hq, hk, hv, ho, hdo, hl, *outs, w.causal, w.scale, best)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ho, hdo, hl))
    d2h = sum(t.numel() * t.element_size() for t in outs)

    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    achieved = flops / (results[best]["main_ms"] / 1e3) / 1e12
    traffic = None
    if os.path.exists(PROFILE_TRAFFIC):
        with open(PROFILE_TRAFFIC) as fh:
            tr = json.load(fh)
        ent = tr.get(w.name, {}).get(best)
        if ent and ent.get("kernel_hash") == kernel_hash():
            traffic = ent["dram_bytes_per_launch"]

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world >= 1:
            cpu = cpu_baseline(w, args.cpu_seconds)
        line = {
            "metric": METRIC, "value": results[best]["tflops"], "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": results[best]["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                       "mask": "causal" if w.causal else "full", "tile": w.tile, "schedule": best,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, outside the step events)",
                       "flops_per_step": flops},
            "pct_bf16_peak": 100.0 * results[best]["tflops"] / world / peak,
            "ratio_vs_atomic": results[best]["vs_atomic"],
            "best_with_extensions": best_with_extensions(results, two_chains, fill, best, world, peak, die, split,
                                                         timed),
            "schedules": results,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic, "kernel": "dash_bwd_main",
                         "peak_source": f"{peak_kind} bf16_tflops (burst)"},
            "e2e": None if not e2e_steps else {"value": world * flops * e2e_steps / e2e_s / 1e12, "unit": "TFLOPS",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": "dash_attn_bwd_host (pinned host buffers)"},
            "workloads": also or None,
            "extension_two_dq_chains": two_chains or None,
            "extension_die_aware": die or None,
            "extension_fill": fill or None,
            "extension_split": split or None,
            "extension_timed": timed or None,
            "runtime_choice": choice,
            "gpu_launches": launches,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
