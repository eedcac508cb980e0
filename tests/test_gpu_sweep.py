"""The pages' sweep on the GPU: 16384 tokens, S = 512 ... 16384, hidden size 2048,
head dimension 64 and 128, both masks (24 configurations, every schedule valid
for the mask).

Each configuration is checked through the C ABI on sampled rows of four heads
(the first, the last and two drawn from a seeded generator): O and LSE at
sampled query rows, dQ at sampled query rows and dK, dV at sampled key rows,
all against the row-wise fp64 oracle, which computes each row from the
definition without forming an S x S matrix.  The rows are the first and last
of the sequence, both sides of a tile boundary, one in the middle, and eight
drawn from the seeded generator per configuration, so that tile-local errors
away from those fixed rows are caught.  Every deterministic schedule must also
give the same bits twice.  Shift or symmetric shift also runs with split gangs
as the library picks them (an extension), to the same checks.
"""
import numpy as np
import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash
import workloads
from oracle import attention as A

from _gpu import LSE_ABS_TOL, assert_close, err

pytestmark = pytest.mark.gpu

SWEEP = workloads.pages_sweep()


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("w", SWEEP, ids=[w.name for w in SWEEP])
def test_pages_sweep_sampled_rows(w):
    dev = torch.device("cuda:0")
    q, k, v, do = (t.to(dev) for t in workloads.make_workload_inputs(w))
    o, lse = dash.attn_fwd(q, k, v, w.causal, w.scale)
    dash.dash_sync_status()
    rng = np.random.default_rng(w.S * 1000 + w.D + (1 if w.causal else 0))
    extra = rng.choice(w.B * w.H, size=min(2, w.B * w.H), replace=False)
    heads = sorted({(0, 0), (w.B - 1, w.H - 1)} | {(int(x) // w.H, int(x) % w.H) for x in extra})
    rows = sorted({0, w.tile - 1, w.tile, w.S // 2 + 5, w.S - 1} | {int(x) for x in rng.integers(0, w.S, 8)})
    refs = {}
    for (b, h) in heads:
        qh, kh, vh, doh = (x[b, h].double().cpu().numpy() for x in (q, k, v, do))
        ro, rl = A.forward_rows(qh, kh, vh, w.causal, w.scale, rows)
        assert_close(f"{w.name} O[{b},{h}] rows", o[b, h][rows], ro)
        assert err(lse[b, h][rows], rl)[1] <= LSE_ABS_TOL
        # the backward is fed the GPU's O and LSE, as the library's callers do
        oh, lh = o[b, h].double().cpu().numpy(), lse[b, h].double().cpu().numpy()
        refs[(b, h)] = A.backward_rows(qh, kh, vh, oh, doh, lh, w.causal, w.scale, rows)
    # every schedule of the mask, and shift / symmetric shift with split gangs as the library picks them
    runs = [(s_, 0) for s_ in w.schedules]
    runs += [(s_, -1) for s_ in ("shift", "symmetric_shift") if s_ in w.schedules]
    for sched, split in runs:
        label = f"{sched} (split gangs)" if split else sched
        first = dash.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, sched, tile=w.tile, shift_split=split)
        dash.dash_sync_status()
        for (b, h), ref in refs.items():
            for name, x, r in zip(("dQ", "dK", "dV"), first, ref):
                assert_close(f"{w.name} {label} {name}[{b},{h}] rows", x[b, h][rows], r)
        assert all(torch.isfinite(x).all() for x in first)
        if sched != "atomic":
            again = dash.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, sched, tile=w.tile, shift_split=split)
            dash.dash_sync_status()
            assert all(torch.equal(a, b) for a, b in zip(first, again)), f"{w.name} {label} not bit-identical"
