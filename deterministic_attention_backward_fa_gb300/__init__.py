"""Python binding of libdash (deterministic attention backward for GB300 / sm_103a).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  The functions named ``dash_*`` mirror the C ABI in include/dash.h
one to one and take torch tensors (device tensors unless stated), passing
their data pointers and the current CUDA stream.  ``attn_fwd`` / ``attn_bwd``
allocate the outputs for convenience.

The library must be built first (``__graft_entry__.build()`` or
``python -m deterministic_attention_backward_fa_gb300._build``); importing a
function without it raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

from . import _build

SCHEDULES = {"atomic": 0, "serial": 1, "descending_q": 2, "shift": 3, "symmetric_shift": 4}
STATUS = {0: "DASH_OK", 1: "DASH_ERR_INVALID_ARG", 2: "DASH_ERR_UNSUPPORTED", 3: "DASH_ERR_CUDA",
          4: "DASH_ERR_TIMEOUT", 5: "DASH_ERR_NO_MEMORY", 6: "DASH_ERR_SCHEDULE"}
TASK_FIRST = 1 << 28
TASK_LAST = 1 << 29
TASK_RANK_MASK = (1 << 24) - 1

# Launches of this library per backward call: preprocess, main, dQ convert.
KERNELS_PER_BWD = 3
KERNELS_PER_FWD = 1


class DashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class BwdOptions(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int), ("num_ctas", ctypes.c_int), ("cost_c", ctypes.c_int),
                ("cost_r", ctypes.c_int), ("spin_limit_ns", ctypes.c_longlong),
                ("dq_accum_out", ctypes.c_void_p), ("tasks", ctypes.c_void_p), ("cta_off", ctypes.c_void_p),
                ("main_begin_event", ctypes.c_void_p), ("main_end_event", ctypes.c_void_p),
                ("dq_chains", ctypes.c_int), ("shift_fill", ctypes.c_int), ("trust_table", ctypes.c_int),
                ("trace", ctypes.c_void_p), ("die_aware", ctypes.c_int), ("cluster_size", ctypes.c_int),
                ("shift_split", ctypes.c_int), ("rank_order", ctypes.c_int)]

# Slots of a trace row (dash_bwd_options_t.trace): see include/dash.h.
TRACE_SLOTS = 21


_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

_SIGS = {
    "dash_attn_fwd": ([_P] * 5 + [_I] * 5 + [_F, _P], _I),
    "dash_attn_fwd_ex": ([_P] * 5 + [_I] * 5 + [_F, _I, _P], _I),
    "dash_attn_bwd": ([_P] * 9 + [_I] * 5 + [_F, _I, _P], _I),
    "dash_attn_bwd_ex": ([_P] * 9 + [_I] * 5 + [_F, _I, ctypes.POINTER(BwdOptions), _P], _I),
    "dash_attn_bwd_host": ([_P] * 9 + [_I] * 5 + [_F, _I, _P], _I),
    "dash_attn_bwd_noalloc": ([_P] * 9 + [_I] * 5 + [_F, _I, _P], _I),
    "dash_schedule_num_tasks": ([_I, _I, _I, _I], ctypes.c_longlong),
    "dash_build_schedule": ([_I, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_build_shift_fill": ([_I] * 7 + [_P, _P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I),
                                          ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_choose_ctas": ([_I] * 7, _I),
    "dash_build_split_schedule": ([_I] * 8 + [_P, _P, ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_build_schedule_ex": ([_I] * 9 + [_P, _P, ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_choose_split_ctas": ([_I] * 8, _I),
    "dash_choose_split": ([_I] * 8 + [ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_choose_schedule_split": ([_I] * 6 + [ctypes.POINTER(_I), ctypes.POINTER(_I),
                                               ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_choose_layout": ([_I] * 6 + [ctypes.POINTER(_I)] * 3 + [ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_check_table": ([_I] * 4 + [_P, _P, _I], _I),
    "dash_fit_costs": ([_I] * 4 + [ctypes.c_double] * 2 + [ctypes.POINTER(_I)] * 2, _I),
    "dash_choose_schedule": ([_I] * 6 + [ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_cluster_latencies": ([_P, _I, _I, _P, _P], _I),
    "dash_place_schedule": ([_P, _P] + [_I] * 5 + [_P, _I, _P, _I, _P, _I, _P, _I, _I, _P, _P], _I),
    "dash_die_map": ([_P, _P, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)], _I),
    "dash_cluster_links": ([_P, _P] + [_I] * 5 + [_P, ctypes.POINTER(ctypes.c_longlong)], _I),
    "dash_sync_status": ([_P], _I),
    "dash_release_workspace": ([], None),
    "dash_last_error": ([], ctypes.c_char_p),
    "dash_version": ([], _I),
}


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libdash.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _LIB = L
    return _LIB


def _check(code: int):
    if code != 0:
        raise DashError(code, lib().dash_last_error().decode())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _shape(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("tensors are [B, H, S, D]")
    return tuple(int(x) for x in q.shape)


def _sched(s) -> int:
    return SCHEDULES[s] if isinstance(s, str) else int(s)


# ------------------------------------------------------------ C mirrors
def dash_attn_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None):
    B, H, S, D = _shape(q)
    bf = torch.bfloat16
    _check(lib().dash_attn_fwd(_dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(o, bf, "o"),
                               _dev(lse, torch.float32, "lse"), B, H, S, D, int(causal), float(scale),
                               _stream(stream)))


def dash_attn_fwd_ex(q, k, v, o, lse, causal: bool, scale: float, cta_pair: int = -1, stream=None):
    """``cta_pair``: 0 = one CTA per Q tile, 1 = CTA-pair (cta_group::2) kernel (D = 128), -1 = default."""
    B, H, S, D = _shape(q)
    bf = torch.bfloat16
    _check(lib().dash_attn_fwd_ex(_dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(o, bf, "o"),
                                  _dev(lse, torch.float32, "lse"), B, H, S, D, int(causal), float(scale),
                                  int(cta_pair), _stream(stream)))


def dash_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, schedule, stream=None):
    B, H, S, D = _shape(q)
    bf = torch.bfloat16
    _check(lib().dash_attn_bwd(_dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(o, bf, "o"),
                               _dev(do, bf, "do"), _dev(lse, torch.float32, "lse"), _dev(dq, bf, "dq"),
                               _dev(dk, bf, "dk"), _dev(dv, bf, "dv"), B, H, S, D, int(causal), float(scale),
                               _sched(schedule), _stream(stream)))


def dash_attn_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, schedule, tile=0,
                     num_ctas=0, cost_c=0, cost_r=0, spin_limit_ns=0, dq_accum_out=None, tasks=None,
                     cta_off=None, main_events=None, stream=None, dq_chains=0, shift_fill=0, trust_table=0,
                     trace=None, die_aware=0, cluster_size=0, shift_split=0, rank_order=0):
    """``main_events``: optional pair of recorded torch.cuda.Event objects (enable_timing) that the
    library records around the main kernel on the call's stream.  ``dq_chains=2`` splits each dQ
    tile's ordered reduction into two chains by rank parity; ``shift_fill=1`` runs some heads of a
    shift backward with the serial schedule on the SMs that whole gangs leave idle (see
    dash_bwd_options_t).  ``trace``: optional int64 device tensor [n_tasks, TRACE_SLOTS] that the traced
    main kernel fills with per-task phase stamps.  ``die_aware=1`` places each gang of a shift schedule
    on one die with its semaphores homed there; ``cluster_size`` (0 or 1 = none; 2, 4, 8, 16) sets the thread-block
    clusters whose ranks hand the dQ turn over through shared memory; ``shift_split=k`` runs each gang of a
    shift or symmetric-shift schedule as k sub-gangs, and ``shift_split=-1`` lets the library pick k by
    simulated makespan; ``rank_order=1`` reduces each dQ tile in the order the simulated schedule reaches
    it (timed ranks; see dash_bwd_options_t)."""
    B, H, S, D = _shape(q)
    bf = torch.bfloat16
    opt = BwdOptions(tile, num_ctas, cost_c, cost_r, spin_limit_ns, None, None, None, None, None, dq_chains,
                     shift_fill, trust_table)
    if main_events is not None:
        opt.main_begin_event = main_events[0].cuda_event
        opt.main_end_event = main_events[1].cuda_event
    keep = []
    if dq_accum_out is not None:
        opt.dq_accum_out = _dev(dq_accum_out, torch.float32, "dq_accum_out").value
    if trace is not None:
        opt.trace = _dev(trace, torch.int64, "trace").value
    opt.die_aware = die_aware
    opt.cluster_size = cluster_size
    opt.shift_split = shift_split
    opt.rank_order = rank_order
    if tasks is not None:
        t = np.ascontiguousarray(tasks, dtype=np.int32)
        o_ = np.ascontiguousarray(cta_off, dtype=np.int32)
        keep += [t, o_]
        opt.tasks = t.ctypes.data
        opt.cta_off = o_.ctypes.data
        opt.num_ctas = len(o_) - 1
    _check(lib().dash_attn_bwd_ex(_dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(o, bf, "o"),
                                  _dev(do, bf, "do"), _dev(lse, torch.float32, "lse"), _dev(dq, bf, "dq"),
                                  _dev(dk, bf, "dk"), _dev(dv, bf, "dv"), B, H, S, D, int(causal),
                                  float(scale), _sched(schedule), ctypes.byref(opt), _stream(stream)))


def dash_attn_bwd_host(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, schedule, stream=None):
    """All tensors are CPU tensors (pinned for full copy bandwidth); blocks until dq/dk/dv are filled."""
    B, H, S, D = _shape(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("lse", lse), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    _check(lib().dash_attn_bwd_host(*(ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, o, do, lse, dq, dk, dv)),
                                    B, H, S, D, int(causal), float(scale), _sched(schedule), _stream(stream)))


def dash_attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale: float, schedule, stream=None):
    """dash_attn_bwd without device allocation (fixed 32 MiB library-owned workspace; synchronises)."""
    B, H, S, D = _shape(q)
    bf = torch.bfloat16
    _check(lib().dash_attn_bwd_noalloc(_dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(o, bf, "o"),
                                       _dev(do, bf, "do"), _dev(lse, torch.float32, "lse"), _dev(dq, bf, "dq"),
                                       _dev(dk, bf, "dk"), _dev(dv, bf, "dv"), B, H, S, D, int(causal),
                                       float(scale), _sched(schedule), _stream(stream)))


def dash_schedule_num_tasks(BH: int, n: int, causal: bool, schedule) -> int:
    return int(lib().dash_schedule_num_tasks(BH, n, int(causal), _sched(schedule)))


def dash_build_schedule(BH: int, n: int, causal: bool, schedule, P: int, cost_c: int = 4, cost_r: int = 1):
    """Host-only.  Returns (tasks int32 [N, 4], cta_off int32 [P+1], makespan)."""
    nt = dash_schedule_num_tasks(BH, n, causal, schedule)
    if nt < 0:
        raise DashError(2, "schedule invalid for this mask / n")
    tasks = np.zeros((max(nt, 1), 4), dtype=np.int32)
    off = np.zeros(P + 1, dtype=np.int32)
    ms = ctypes.c_longlong(0)
    _check(lib().dash_build_schedule(BH, n, int(causal), _sched(schedule), P, cost_c, cost_r,
                                     tasks.ctypes.data_as(ctypes.c_void_p), off.ctypes.data_as(ctypes.c_void_p),
                                     ctypes.byref(ms)))
    return tasks[:nt], off, int(ms.value)


def dash_build_shift_fill(BH: int, n: int, causal: bool, schedule, max_ctas: int, cost_c: int = 4, cost_r: int = 1):
    """Host-only.  Returns (tasks int32 [N, 4], cta_off int32 [P+1], P, shift_heads, fill schedule name or
    None, makespan)."""
    nt = dash_schedule_num_tasks(BH, n, causal, schedule)
    if nt < 0:
        raise DashError(2, "schedule invalid for this mask / n")
    tasks = np.zeros((max(nt, 1), 4), dtype=np.int32)
    off = np.zeros(max_ctas + 1, dtype=np.int32)
    P, hs, fm, ms = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(-1), ctypes.c_longlong(0)
    _check(lib().dash_build_shift_fill(BH, n, int(causal), _sched(schedule), max_ctas, cost_c, cost_r,
                                       tasks.ctypes.data_as(ctypes.c_void_p), off.ctypes.data_as(ctypes.c_void_p),
                                       ctypes.byref(P), ctypes.byref(hs), ctypes.byref(fm), ctypes.byref(ms)))
    fill = next(k for k, v in SCHEDULES.items() if v == fm.value) if fm.value >= 0 else None
    return tasks[:nt], off[:P.value + 1], int(P.value), int(hs.value), fill, int(ms.value)


def dash_check_table(BH: int, n: int, causal: bool, tasks, cta_off, dq_chains: int = 0):
    """Host-only.  Raises DashError (code 6) if the table's dQ orders could not finish."""
    t = np.ascontiguousarray(tasks, dtype=np.int32).reshape(-1, 4)
    o = np.ascontiguousarray(cta_off, dtype=np.int32)
    _check(lib().dash_check_table(BH, n, int(causal), dq_chains, t.ctypes.data_as(ctypes.c_void_p),
                                  o.ctypes.data_as(ctypes.c_void_p), len(o) - 1))


def dash_fit_costs(BH: int, n: int, causal: bool, max_ctas: int, atomic_ms: float, serial_ms: float):
    """Host-only.  Returns (cost_c, cost_r) fitted to the measured atomic and serial times."""
    c, r = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().dash_fit_costs(BH, n, int(causal), max_ctas, float(atomic_ms), float(serial_ms), ctypes.byref(c),
                                ctypes.byref(r)))
    return int(c.value), int(r.value)


def dash_choose_ctas(BH: int, n: int, causal: bool, schedule, max_ctas: int, cost_c: int = 4, cost_r: int = 1):
    return int(lib().dash_choose_ctas(BH, n, int(causal), _sched(schedule), max_ctas, cost_c, cost_r))


def dash_build_schedule_ex(BH: int, n: int, causal: bool, schedule, split: int, rank_order: int, P: int,
                           cost_c: int = 4, cost_r: int = 1):
    """Host-only tables with split gangs and / or timed ranks.  Returns (tasks int32 [N, 4], cta_off int32 [P+1],
    makespan)."""
    nt = dash_schedule_num_tasks(BH, n, causal, schedule)
    if nt < 0:
        raise DashError(2, "schedule invalid for this mask / n")
    tasks = np.zeros((max(nt, 1), 4), dtype=np.int32)
    off = np.zeros(P + 1, dtype=np.int32)
    ms = ctypes.c_longlong(0)
    _check(lib().dash_build_schedule_ex(BH, n, int(causal), _sched(schedule), split, rank_order, P, cost_c, cost_r,
                                        tasks.ctypes.data, off.ctypes.data, ctypes.byref(ms)))
    return tasks[:nt], off, ms.value


def dash_build_split_schedule(BH: int, n: int, causal: bool, schedule, split: int, P: int, cost_c: int = 4,
                              cost_r: int = 1):
    """Host-only split-gang tables (an extension).  Returns (tasks int32 [N, 4], cta_off int32 [P+1], makespan)."""
    nt = dash_schedule_num_tasks(BH, n, causal, schedule)
    if nt < 0:
        raise DashError(2, "schedule invalid for this mask / n")
    tasks = np.zeros((max(nt, 1), 4), dtype=np.int32)
    off = np.zeros(P + 1, dtype=np.int32)
    ms = ctypes.c_longlong(0)
    _check(lib().dash_build_split_schedule(BH, n, int(causal), _sched(schedule), split, P, cost_c, cost_r,
                                           tasks.ctypes.data, off.ctypes.data, ctypes.byref(ms)))
    return tasks[:nt], off, ms.value


def dash_choose_split(BH: int, n: int, causal: bool, schedule, max_ctas: int, num_ctas: int = 0, cost_c: int = 4,
                      cost_r: int = 1):
    """Host-only.  The split that ``shift_split=-1`` picks: returns (k, CTA count, simulated makespan), k = -1
    where split gangs do not apply."""
    P, ms = _I(0), ctypes.c_longlong(0)
    k = lib().dash_choose_split(BH, n, int(causal), _sched(schedule), max_ctas, num_ctas, cost_c, cost_r,
                                ctypes.byref(P), ctypes.byref(ms))
    return int(k), P.value, ms.value


def dash_choose_split_ctas(BH: int, n: int, causal: bool, schedule, split: int, max_ctas: int, cost_c: int = 4,
                           cost_r: int = 1):
    return int(lib().dash_choose_split_ctas(BH, n, int(causal), _sched(schedule), split, max_ctas, cost_c, cost_r))


def dash_choose_schedule_split(BH: int, n: int, causal: bool, max_ctas: int, cost_c: int = 4, cost_r: int = 1):
    """Host-only.  ``dash_choose_schedule`` with split gangs among the candidates.  Returns (schedule name, CTA
    count, split, simulated makespan)."""
    P, k, ms = _I(0), _I(0), ctypes.c_longlong(0)
    s = lib().dash_choose_schedule_split(BH, n, int(causal), max_ctas, cost_c, cost_r, ctypes.byref(P),
                                         ctypes.byref(k), ctypes.byref(ms))
    if s < 0:
        raise DashError(1, dash_last_error())
    return {v: k_ for k_, v in SCHEDULES.items()}[s], P.value, k.value, ms.value


def dash_choose_layout(BH: int, n: int, causal: bool, max_ctas: int, cost_c: int = 4, cost_r: int = 1):
    """Host-only.  The runtime choice over every deterministic layout: returns (schedule name, CTA count, split,
    rank_order, simulated makespan)."""
    P, k, ro, ms = _I(0), _I(0), _I(0), ctypes.c_longlong(0)
    s = lib().dash_choose_layout(BH, n, int(causal), max_ctas, cost_c, cost_r, ctypes.byref(P), ctypes.byref(k),
                                 ctypes.byref(ro), ctypes.byref(ms))
    if s < 0:
        raise DashError(1, dash_last_error())
    return {v: k_ for k_, v in SCHEDULES.items()}[s], P.value, k.value, ro.value, ms.value


def dash_choose_schedule(BH: int, n: int, causal: bool, max_ctas: int, cost_c: int = 4, cost_r: int = 1):
    """Host-only.  Returns (schedule name, CTA count, simulated makespan) of the
    deterministic schedule with the smallest simulated makespan."""
    P, ms = _I(0), ctypes.c_longlong(0)
    s = lib().dash_choose_schedule(BH, n, int(causal), max_ctas, cost_c, cost_r, ctypes.byref(P), ctypes.byref(ms))
    if s < 0:
        raise DashError(1, dash_last_error())
    return {v: k for k, v in SCHEDULES.items()}[s], P.value, ms.value


def dash_cluster_latencies(lat):
    """Host-only.  lat: [n_sms, n_lines] latencies (clocks).  Returns (group per SM, home per line)."""
    L = np.ascontiguousarray(lat, dtype=np.uint32)
    g = np.zeros(L.shape[0], dtype=np.int32)
    h = np.zeros(L.shape[1], dtype=np.int32)
    _check(lib().dash_cluster_latencies(L.ctypes.data_as(ctypes.c_void_p), L.shape[0], L.shape[1],
                                        g.ctypes.data_as(ctypes.c_void_p), h.ctypes.data_as(ctypes.c_void_p)))
    return g, h


def dash_place_schedule(tasks, cta_off, gang: int, BH: int, n: int, chains: int, smids, lines, max_smid: int):
    """Host-only.  smids, lines: pairs of int lists (group 0, group 1).  Returns (slot_of_smid, sem_idx)."""
    t = np.ascontiguousarray(tasks, dtype=np.int32).reshape(-1, 4)
    o = np.ascontiguousarray(cta_off, dtype=np.int32)
    a = [np.ascontiguousarray(x, dtype=np.int32) for x in (*smids, *lines)]
    slot = np.zeros(max_smid + 1, dtype=np.int32)
    sem = np.zeros(BH * n * chains, dtype=np.int32)
    p = lambda x: x.ctypes.data_as(ctypes.c_void_p)
    _check(lib().dash_place_schedule(p(t), p(o), len(o) - 1, gang, BH, n, chains, p(a[0]), len(a[0]), p(a[1]),
                                     len(a[1]), p(a[2]), len(a[2]), p(a[3]), len(a[3]), max_smid, p(slot), p(sem)))
    return slot, sem


def dash_cluster_links(tasks, cta_off, C: int, BH: int, n: int, chains: int = 1):
    """Host-only.  Returns (link word per task, number of linked hand-offs) for clusters of C."""
    t = np.ascontiguousarray(tasks, dtype=np.int32).reshape(-1, 4)
    o = np.ascontiguousarray(cta_off, dtype=np.int32)
    out = np.zeros(len(t), dtype=np.int32)
    k = ctypes.c_longlong(0)
    _check(lib().dash_cluster_links(t.ctypes.data_as(ctypes.c_void_p), o.ctypes.data_as(ctypes.c_void_p),
                                    len(o) - 1, C, BH, n, chains, out.ctypes.data_as(ctypes.c_void_p),
                                    ctypes.byref(k)))
    return out, int(k.value)


def dash_die_map(max_sm: int = 1023, stream=None):
    """The device's SM groups as the stream's workspace measures them: (group per SM id, -1 for ids the
    device does not have; n0, n1)."""
    g = np.zeros(max_sm + 1, dtype=np.int32)
    n0, n1 = _I(0), _I(0)
    _check(lib().dash_die_map(_stream(stream), g.ctypes.data_as(ctypes.c_void_p), max_sm, ctypes.byref(n0),
                              ctypes.byref(n1)))
    return g, n0.value, n1.value


def dash_sync_status(stream=None):
    _check(lib().dash_sync_status(_stream(stream)))


def dash_release_workspace():
    lib().dash_release_workspace()


def dash_last_error() -> str:
    return lib().dash_last_error().decode()


def dash_version() -> int:
    return int(lib().dash_version())


# ------------------------------------------------------------ conveniences
def attn_fwd(q, k, v, causal: bool, scale: float | None = None, stream=None, cta_pair: int = -1):
    """O (bf16) and LSE (fp32, natural log) of softmax attention."""
    B, H, S, D = _shape(q)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if cta_pair == -1:
        dash_attn_fwd(q, k, v, o, lse, causal, scale, stream)
    else:
        dash_attn_fwd_ex(q, k, v, o, lse, causal, scale, cta_pair, stream)
    return o, lse


def attn_bwd(q, k, v, o, do, lse, causal: bool, scale: float | None = None, schedule="serial",
             dq_accum: bool = False, stream=None, **opts):
    """dQ, dK, dV (bf16); with ``dq_accum`` also the unscaled fp32 dQ accumulator."""
    B, H, S, D = _shape(q)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    acc = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq_accum else None
    if acc is None and not opts:
        dash_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, causal, scale, schedule, stream)
    else:
        dash_attn_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, causal, scale, schedule, dq_accum_out=acc,
                         stream=stream, **opts)
    return (dq, dk, dv, acc) if dq_accum else (dq, dk, dv)
