"""The allocation-free backward, dash_attn_bwd_noalloc.

Some callers cannot allocate device memory while they run: a framework whose
caching allocator owns all of the GPU's memory, or a runtime that reserves a
fixed memory budget up front.  This entry point serves them with a fixed
scratch array inside the library.  These tests call it through the C ABI
twice in a row (the second call finds the scratch as the first one left it)
and check each result against the fp64 oracle within the parity tolerance of
the other GPU tests, and against dash_attn_bwd on the same inputs: within
that tolerance, and bit for bit, since both run the same kernels with the
same deterministic schedule table.  The file sorts last so that a run which
stops at the first failure has run every other test before this one.
"""
import ctypes

import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash
from oracle import attention as A

from _gpu import ABS_TOL, REL_TOL, Problem, assert_close


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,S,D,causal,sched", [(2, 4, 1000, 128, True, "descending_q"),
                                                  (2, 4, 1024, 128, True, "symmetric_shift"),
                                                  (1, 3, 512, 64, False, "shift"),
                                                  (1, 2, 256, 64, True, "serial")])
def test_noalloc_matches_oracle_and_allocating_entry_point_twice(B, H, S, D, causal, sched):
    P = Problem(B, H, S, D, causal)
    o, lse = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale)
    ref = dash.attn_bwd(P.q, P.k, P.v, o, P.do, lse, causal, P.scale, sched)
    dash.dash_sync_status()
    q, k, v, do = P.f64
    ro, rl = A.forward(q, k, v, causal, P.scale)
    oracle = A.backward(q, k, v, ro, do, rl, causal, P.scale)   # end to end: oracle forward and backward
    for call in range(2):   # the second call reuses the scratch the first one left behind
        outs = [torch.full_like(P.q, float("nan")) for _ in range(3)]
        dash.dash_attn_bwd_noalloc(P.q, P.k, P.v, o, P.do, lse, *outs, causal, P.scale, sched)
        for name, x, r, orc in zip(("dQ", "dK", "dV"), outs, ref, oracle):
            assert_close(f"call {call}: noalloc {name} against the oracle", x, orc)
            assert_close(f"call {call}: noalloc {name} against dash_attn_bwd", x.float(),
                         r.double().cpu().numpy(), rel=REL_TOL, abs_=ABS_TOL)
            assert torch.equal(x, r), f"call {call}: noalloc {name} differs in bits from dash_attn_bwd"


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch():
    P = Problem(1, 1, 128, 64, False)
    big = dash.lib().dash_attn_bwd_noalloc(*([ctypes.c_void_p(P.q.data_ptr())] * 9), 8, 32, 8192, 128, 0,
                                           0.1, 1, ctypes.c_void_p(0))
    assert big == 2
    assert "scratch" in dash.dash_last_error()


def test_noalloc_size_check_needs_no_gpu():
    # the size checks come before any CUDA call, so they run on a machine without a GPU
    fake = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced
    rc = dash.lib().dash_attn_bwd_noalloc(*([fake] * 9), 4, 32, 16384, 128, 1, 0.1, 1, ctypes.c_void_p(0))
    assert rc == 2
    assert "scratch" in dash.dash_last_error()
    rc = dash.lib().dash_attn_bwd_noalloc(*([fake] * 9), 1 << 16, 1 << 16, 128, 128, 1, 0.1, 1,
                                          ctypes.c_void_p(0))
    assert rc == 1
    assert "too large" in dash.dash_last_error()
