"""The allocation-free backward, dash_attn_bwd_noalloc.

It serves callers that must not allocate device memory while they run (a
framework whose caching allocator owns the GPU's memory, a runtime with a
fixed budget reserved up front): its workspace is a fixed array inside the
library.  These tests call it through the C ABI twice in a row and compare
each result with dash_attn_bwd's on the same inputs, within the parity
tolerance of the other GPU tests.  The file sorts last so that a run which
stops at the first failure has run every other test before this one.
"""
import ctypes

import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash

from _gpu import ABS_TOL, REL_TOL, Problem, assert_close


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,S,D,causal,sched", [(2, 4, 1000, 128, True, "symmetric_shift"),
                                                  (1, 3, 512, 64, False, "shift"),
                                                  (1, 2, 256, 64, True, "serial")])
def test_noalloc_matches_allocating_entry_point_twice(B, H, S, D, causal, sched):
    if sched == "symmetric_shift" and ((S + 127) // 128) % 2:
        sched = "descending_q"
    P = Problem(B, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    ref = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched)
    dash.dash_sync_status()
    for _ in range(2):   # the second call reuses the scratch the first one left behind
        outs = [torch.full_like(P.q, float("nan")) for _ in range(3)]
        dash.dash_attn_bwd_noalloc(P.q, P.k, P.v, o, P.do, lse, *outs, causal, P.scale, sched)
        for name, x, r in zip(("dQ", "dK", "dV"), outs, ref):
            assert_close(f"noalloc {name}", x.float(), r.double().cpu().numpy(), rel=REL_TOL, abs_=ABS_TOL)


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch():
    P = Problem(1, 1, 128, 64, False)
    big = dash.lib().dash_attn_bwd_noalloc(*([ctypes.c_void_p(P.q.data_ptr())] * 9), 8, 32, 8192, 128, 0,
                                           0.1, 1, ctypes.c_void_p(0))
    assert big == 2
    assert "scratch" in dash.dash_last_error()


def test_noalloc_size_check_needs_no_gpu():
    # the size check comes before any CUDA call, so it runs on a machine without a GPU
    fake = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced
    rc = dash.lib().dash_attn_bwd_noalloc(*([fake] * 9), 4, 32, 16384, 128, 1, 0.1, 1, ctypes.c_void_p(0))
    assert rc == 2
    assert "scratch" in dash.dash_last_error()
