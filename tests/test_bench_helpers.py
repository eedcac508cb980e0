"""Host-side helpers of bench.py (no GPU): the fastest deterministic layout
including the extensions, and the runtime schedule choice with fitted costs."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import deterministic_attention_backward_fa_gb300 as dash  # noqa: E402
import workloads  # noqa: E402


def test_best_with_extensions_picks_the_fastest_layout():
    res = {"atomic": {"tflops": 900.0, "vs_atomic": 1.0}, "serial": {"tflops": 600.0, "vs_atomic": 0.667},
           "shift": {"tflops": 750.0, "vs_atomic": 0.833}}
    two = {"shift": {"tflops": 800.0, "vs_atomic": 0.889}}
    fill = {"shift": {"tflops": 850.0, "vs_atomic": 0.944}}
    b = bench.best_with_extensions(res, two, fill, "shift", 1, 2000.0)
    assert b["schedule"] == "shift+fill" and b["tflops"] == 850.0 and abs(b["pct_bf16_peak"] - 42.5) < 1e-9
    b = bench.best_with_extensions(res, two, {}, "shift", 1, 2000.0)
    assert b["schedule"] == "shift+two_dq_chains"
    b = bench.best_with_extensions(res, {}, {}, "shift", 2, 2000.0)   # whole-job value over two GPUs
    assert b["schedule"] == "shift" and abs(b["pct_bf16_peak"] - 18.75) < 1e-9
    split = {"shift": {"tflops": 870.0, "vs_atomic": 0.967, "split": 4}}
    b = bench.best_with_extensions(res, two, fill, "shift", 1, 2000.0, split=split)
    assert b["schedule"] == "shift+split" and b["tflops"] == 870.0
    timed = {"shift": {"tflops": 880.0, "vs_atomic": 0.978}}
    b = bench.best_with_extensions(res, two, fill, "shift", 1, 2000.0, split=split, timed=timed)
    assert b["schedule"] == "shift+timed" and b["tflops"] == 880.0


def test_split_of_needs_a_divisor_of_the_gang():
    full, causal = workloads.WORKLOADS["full_s4096_d128"], workloads.WORKLOADS["causal_s8192_d64"]
    assert bench.split_of(full, "shift", 4) == 4             # a gang of 32 chains
    assert bench.split_of(full, "shift", 3) == 0
    assert bench.split_of(full, "shift", 1) == 0             # 1 = whole gangs, not timed as an extension
    assert bench.split_of(full, "serial", 4) == 0
    assert bench.split_of(full, "symmetric_shift", 4) == 0   # not a schedule of the full mask
    assert bench.split_of(full, "shift", -1) == -1           # the library's choice
    assert bench.split_of(full, "serial", -1) == 0
    assert bench.split_chosen(dash, full, "shift", -1, 152) == dash.dash_choose_split(32, 32, False, "shift", 152)[0]
    assert bench.split_chosen(dash, full, "shift", 4, 152) == 4
    n = causal.S // causal.tile
    assert bench.split_of(causal, "symmetric_shift", 4) == (4 if (n // 2) % 4 == 0 else 0)


def test_best_label_names_split_gangs_only_when_split():
    det = {"serial": 600.0, "shift": 770.0}
    assert bench.best_label(det, {"shift": (870.0, 4)}) == "shift+split"
    assert bench.best_label(det, {"shift": (780.0, 1)}) == "shift"     # k = 1 is whole gangs: no label of its own
    assert bench.best_label(det, {}) == "shift"
    assert bench.best_label(det, {"shift": (870.0, 4)}, {"shift": 880.0}) == "shift+timed"


def test_runtime_choice_uses_the_fitted_costs():
    import __graft_entry__
    __graft_entry__.build()
    w = workloads.WORKLOADS["full_s4096_d128"]
    BH, n = w.B * w.H, w.S // w.tile
    ch = bench.runtime_choice(dash, w, 152, 1.0, 1.45, "shift")
    c, r = dash.dash_fit_costs(BH, n, w.causal, 152, 1.0, 1.45)
    assert (ch["cost_c"], ch["cost_r"]) == (c, r)
    name, ctas, _ = dash.dash_choose_schedule(BH, n, w.causal, 152, c, r)
    assert (ch["chosen"], ch["ctas"]) == (name, ctas)
    assert ch["agrees"] == (name == "shift")
    ch = bench.runtime_choice(dash, w, 152, 1.0, 1.45, "shift", "shift+split")
    name, ctas, k, _ = dash.dash_choose_schedule_split(BH, n, w.causal, 152, c, r)
    assert ch["with_split"]["chosen"] == (f"{name}+split" if k > 1 else name) and ch["with_split"]["split"] == k
    ch = bench.runtime_choice(dash, w, 152, 1.0, 1.45, "shift", "shift+split", "shift+split")
    name, ctas, k, ro, _ = dash.dash_choose_layout(BH, n, w.causal, 152, c, r)
    assert ch["layout"]["chosen"] == name + ("+split" if k > 1 else "") + ("+timed" if ro else "")
