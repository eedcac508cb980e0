"""Pins for the fp64 attention oracle (CPU only).

Each check ties the oracle to something other than itself: central finite
differences of the scalar loss L = sum(O * dO) through the oracle's own
forward, PyTorch's fp64 scaled-dot-product attention with its autograd,
closed-form special cases and invariants that follow from the softmax
definition.  A dropped term, a sign error or a transposed operand anywhere in
forward() or backward() fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def loss(q, k, v, do, causal, scale):
    o, _ = A.forward(q, k, v, causal, scale)
    return float((o * do).sum())


@pytest.mark.parametrize("S,D", [(4, 4), (8, 8), (5, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(S, D, causal):
    B, H = 1, 1
    q, k, v, do = (rnd((B, H, S, D), 10 + i) for i in range(4))
    scale = 1.0 / math.sqrt(D)
    o, lse = A.forward(q, k, v, causal, scale)
    grads = A.backward(q, k, v, o, do, lse, causal, scale)
    h = 1e-6
    for which, g in zip(range(3), grads):
        fd = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd[idx] = (loss(*args_p, do, causal, scale) - loss(*args_m, do, causal, scale)) / (2 * h)
        rel = np.linalg.norm(fd - g) / max(np.linalg.norm(fd), 1e-300)
        assert rel <= 1e-6, (which, rel)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_and_autograd_fp64(causal):
    B, H, S, D = 2, 3, 37, 16
    scale = 0.3
    q, k, v, do = (rnd((B, H, S, D), 20 + i) for i in range(4))
    o, lse = A.forward(q, k, v, causal, scale)
    dq, dk, dv = A.backward(q, k, v, o, do, lse, causal, scale)

    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do, dtype=torch.float64))
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_single_key_closed_form():
    # S = 1: softmax over one key is 1, so O = V, LSE = s, and the score
    # gradient vanishes (dQ = dK = 0) while dV = dO.
    B, H, S, D = 2, 2, 1, 8
    q, k, v, do = (rnd((B, H, S, D), 30 + i) for i in range(4))
    scale = 0.7
    for causal in (False, True):
        o, lse = A.forward(q, k, v, causal, scale)
        np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, scale * (q * k).sum(-1), rtol=1e-14)
        dq, dk, dv = A.backward(q, k, v, o, do, lse, causal, scale)
        assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
        np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)


def test_zero_queries_give_uniform_attention():
    # q = 0: all scores are 0, so P is uniform over the visible keys.
    B, H, S, D = 1, 2, 9, 4
    k, v = rnd((B, H, S, D), 40), rnd((B, H, S, D), 41)
    q = np.zeros((B, H, S, D))
    o, lse = A.forward(q, k, v, False, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, np.full(lse.shape, math.log(S)), rtol=1e-14)
    o, lse = A.forward(q, k, v, True, 1.0)
    cnt = np.arange(1, S + 1)
    np.testing.assert_allclose(o, np.cumsum(v, axis=2) / cnt[:, None], atol=1e-14)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(cnt), lse.shape), rtol=1e-14)


def test_causal_first_row_and_zero_upstream_gradient():
    B, H, S, D = 1, 1, 12, 8
    q, k, v, do = (rnd((B, H, S, D), 50 + i) for i in range(4))
    o, lse = A.forward(q, k, v, True, 0.5)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-15)
    dq, dk, dv = A.backward(q, k, v, o, do, lse, True, 0.5)
    assert np.abs(dq[:, :, 0]).max() < 1e-14          # query 0 sees one key only
    z = A.backward(q, k, v, o, np.zeros_like(do), lse, True, 0.5)
    assert all(np.abs(x).max() == 0 for x in z)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_gradient_invariants(causal):
    B, H, S, D = 2, 2, 19, 8
    q, k, v, do = (rnd((B, H, S, D), 60 + i, 1.5) for i in range(4))
    scale = 1 / math.sqrt(D)
    o, lse = A.forward(q, k, v, causal, scale)
    dq, dk, dv, it = A.backward(q, k, v, o, do, lse, causal, scale, return_intermediates=True)
    ds, p = it["dS"], it["P"]
    # each row of P sums to one, so each row of dS sums to zero
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-13)
    assert np.abs(ds.sum(-1)).max() <= 1e-12 * np.abs(ds).max()
    # hence sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0
    assert np.abs(dk.sum(axis=2)).max() <= 1e-12 * np.abs(dk).max() * S
    # and sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=1e-12, atol=1e-12)
    # delta_i = O_i . dO_i equals sum_j P_ij dP_ij (dP = dO V^T)
    dp = np.einsum("bhid,bhjd->bhij", do, v)
    np.testing.assert_allclose(it["delta"], (p * dp).sum(-1), rtol=1e-11, atol=1e-12)


def test_head_subset_equals_full():
    B, H, S, D = 2, 3, 16, 8
    q, k, v, do = (rnd((B, H, S, D), 70 + i) for i in range(4))
    o, lse = A.forward(q, k, v, True, 0.4)
    full = A.backward(q, k, v, o, do, lse, True, 0.4)
    sub = A.backward_heads(q, k, v, o, do, lse, True, 0.4, [(1, 2), (0, 1)])
    for (b, h), g in sub.items():
        for x, y in zip(g, full):
            np.testing.assert_array_equal(x, y[b, h])


@pytest.mark.parametrize("causal", [False, True])
def test_row_oracle_matches_torch_autograd_and_full_backward(causal):
    # the row-wise forms serve heads too long to form whole; pin them against
    # PyTorch's fp64 attention and autograd, and against the whole-matrix oracle
    S, D = 41, 16
    scale = 0.35
    q, k, v, do = (rnd((1, 1, S, D), 80 + i) for i in range(4))
    rows = [0, 1, 20, 39, 40]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do, dtype=torch.float64))
    o, lse = A.forward(q, k, v, causal, scale)
    ro, rl = A.forward_rows(q[0, 0], k[0, 0], v[0, 0], causal, scale, rows)
    np.testing.assert_allclose(ro, to.detach().numpy()[0, 0][rows], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(rl, lse[0, 0][rows], rtol=1e-13, atol=1e-13)
    rq, rk, rv = A.backward_rows(q[0, 0], k[0, 0], v[0, 0], o[0, 0], do[0, 0], lse[0, 0], causal, scale, rows)
    for got, grad in zip((rq, rk, rv), (tq.grad, tk.grad, tv.grad)):
        np.testing.assert_allclose(got, grad.numpy()[0, 0][rows], rtol=1e-9, atol=1e-11)
    full = A.backward(q, k, v, o, do, lse, causal, scale)
    for got, f in zip((rq, rk, rv), full):
        np.testing.assert_allclose(got, f[0, 0][rows], rtol=1e-12, atol=1e-13)
