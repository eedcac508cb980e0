"""The CTA-pair forward (dash_attn_fwd_ex with cta_pair = 1): two CTAs of a
cluster share every M = 256 tcgen05 MMA (cta_group::2), each loading half of
the K and V tiles.  O and LSE must meet the parity bar against the fp64
oracle, on even and odd numbers of Q tiles (the last pair then has a CTA whose
rows are all past the sequence) and ragged tails, and agree with the
single-CTA forward within rounding."""
import numpy as np
import pytest
import torch

import deterministic_attention_backward_fa_gb300 as dash

from _gpu import LSE_ABS_TOL, Problem, assert_close, err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


PAIR_CASES = [(1, 2, 512, True), (1, 2, 512, False), (2, 3, 640, True), (1, 1, 100, True), (1, 1, 1000, False),
              (1, 4, 2048, True), (1, 2, 384, False)]


@pytest.mark.parametrize("B,H,S,causal", PAIR_CASES)
def test_pair_forward_matches_oracle_and_single_cta(B, H, S, causal):
    P = Problem(B, H, S, 128, causal)
    o2, l2 = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale, cta_pair=1)
    o1, l1 = dash.attn_fwd(P.q, P.k, P.v, causal, P.scale, cta_pair=0)
    dash.dash_sync_status()
    ro, rl = P.oracle_fwd()
    assert_close("pair O", o2, ro)
    assert err(l2, rl)[1] <= LSE_ABS_TOL
    assert_close("pair O vs single-CTA O", o2, o1.double().cpu().numpy())
    assert float((l2 - l1).abs().max()) <= 1e-4
    # the backward runs on the pair forward's outputs like on any other
    dq, dk, dv = dash.attn_bwd(P.q, P.k, P.v, o2, P.do, l2, causal, P.scale, "serial")
    dash.dash_sync_status()
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()


def test_pair_forward_needs_d128():
    P = Problem(1, 1, 256, 64, False)
    o = torch.empty_like(P.q)
    lse = torch.empty((1, 1, 256), dtype=torch.float32, device=P.q.device)
    with pytest.raises(dash.DashError) as ei:
        dash.dash_attn_fwd_ex(P.q, P.k, P.v, o, lse, False, P.scale, 1)
    assert ei.value.code == 2
