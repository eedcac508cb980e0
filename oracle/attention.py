"""fp64 CPU oracle for softmax attention, forward and backward.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline may import this module; the library never does, and this module
imports nothing from the library.

What it computes.  The DASH write-ups take the FlashAttention backward as given
(DASH overview (zskr.cn), section 2.1: each SM computes partial dQ/dK/dV for
its tile and dQ is reduced globally; Sintesi Tecnica DASH (gist.science/it),
section 1: the accumulation order of dQ must be fixed).  They never write the
attention equations out, so this oracle is the textbook definition of softmax
attention and its gradient, per (batch, head), in float64:

    s_ij   = scale * q_i . k_j            (s_ij = -inf when causal and j > i)
    LSE_i  = log sum_j exp(s_ij)          (natural log, scale inside)
    P_ij   = exp(s_ij - LSE_i)
    O_i    = sum_j P_ij v_j
    dV_j   = sum_i P_ij dO_i
    dP_ij  = dO_i . v_j
    delta_i= sum_d dO_id O_id
    dS_ij  = P_ij (dP_ij - delta_i)
    dQ_i   = scale * sum_j dS_ij k_j
    dK_j   = scale * sum_i dS_ij q_i

Inputs are float64 numpy arrays of shape [B, H, S, D] (bf16 values widened
exactly by the caller).  Causal masking is square and top-left aligned: query
i sees keys j <= i.  Every matrix is formed whole, per head; numpy's matmul is
the only library primitive used.

Pins (tests/test_oracle.py): central finite differences of L = sum(O * dO),
PyTorch's fp64 scaled-dot-product attention and its autograd on CPU,
closed-form special cases (S = 1, q = 0, causal row 0), and invariants
(rows of dS sum to zero, sum_j dK_j = 0, sum_j dV_j = sum_i dO_i).  The
row-wise forms (``forward_rows``, ``backward_rows``), which check heads too
long to form whole one row at a time, are pinned to PyTorch's autograd too.
"""
from __future__ import annotations

import numpy as np


def _scores(q, k, scale, causal):
    """s = scale * q k^T with the causal mask applied as -inf."""
    s = scale * (q @ k.T)
    if causal:
        S = s.shape[0]
        s[np.triu_indices(S, k=1)] = -np.inf
    return s


def forward(q, k, v, causal: bool, scale: float):
    """Softmax attention forward.  Returns (O [B,H,S,D], LSE [B,H,S]), fp64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, S, D = q.shape
    o = np.empty((B, H, S, D))
    lse = np.empty((B, H, S))
    for b in range(B):
        for h in range(H):
            s = _scores(q[b, h], k[b, h], scale, causal)
            m = s.max(axis=1, keepdims=True)          # finite: j = i is never masked
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)
            lse[b, h] = (m + np.log(l))[:, 0]
            o[b, h] = (e / l) @ v[b, h]
    return o, lse


def backward(q, k, v, o, do, lse, causal: bool, scale: float, return_intermediates: bool = False):
    """Softmax attention backward from (Q, K, V, O, dO, LSE).

    Returns (dQ, dK, dV), each [B,H,S,D] fp64.  With ``return_intermediates``
    it also returns a dict holding P, dS (per head, [B,H,S,S]) and delta
    ([B,H,S]) so that the tests can check their invariants; only use that on
    small shapes.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    B, H, S, D = q.shape
    dq = np.empty((B, H, S, D))
    dk = np.empty((B, H, S, D))
    dv = np.empty((B, H, S, D))
    inter = {"P": np.empty((B, H, S, S)), "dS": np.empty((B, H, S, S)),
             "delta": np.empty((B, H, S))} if return_intermediates else None
    for b in range(B):
        for h in range(H):
            s = _scores(q[b, h], k[b, h], scale, causal)
            p = np.exp(s - lse[b, h][:, None])        # exp(-inf) = 0 on masked entries
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            delta = (do[b, h] * o[b, h]).sum(axis=1)
            ds = p * (dp - delta[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
            if inter is not None:
                inter["P"][b, h] = p
                inter["dS"][b, h] = ds
                inter["delta"][b, h] = delta
    if inter is not None:
        return dq, dk, dv, inter
    return dq, dk, dv


def backward_heads(q, k, v, o, do, lse, causal: bool, scale: float, heads):
    """Backward restricted to the listed (b, h) pairs: each head is independent,
    so this is ``backward`` evaluated on a subset.  Returns a dict
    {(b, h): (dQ, dK, dV)} with [S, D] fp64 arrays."""
    out = {}
    for (b, h) in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        r = backward(q[sl], k[sl], v[sl], o[sl], do[sl], lse[sl], causal, scale)
        out[(b, h)] = tuple(x[0, 0] for x in r)
    return out


def forward_heads(q, k, v, causal: bool, scale: float, heads):
    """Forward restricted to the listed (b, h) pairs: {(b, h): (O [S,D], LSE [S])}."""
    out = {}
    for (b, h) in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        o, lse = forward(q[sl], k[sl], v[sl], causal, scale)
        out[(b, h)] = (o[0, 0], lse[0, 0])
    return out


def flops_fp64(B, H, S, D, causal: bool) -> float:
    """Floating-point work the oracle's backward spends (five S x S x D
    matmuls per head, counted 2 flops per multiply-add; the causal case is
    counted at the full-matrix cost because the oracle forms whole matrices)."""
    return 10.0 * B * H * S * S * D


def forward_rows(q, k, v, causal: bool, scale: float, rows):
    """O and LSE of one head ([S, D] fp64 inputs) at the listed query rows only,
    each row from the definition in the module docstring (O(S*D) per row, so it
    serves heads too long to form whole).  Returns (O [len(rows), D], LSE [len(rows)])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S, D = q.shape
    o = np.empty((len(rows), D))
    lse = np.empty(len(rows))
    for r, i in enumerate(rows):
        s = scale * (k @ q[i])                      # s_ij over all keys j
        if causal:
            s[i + 1:] = -np.inf
        m = s.max()
        e = np.exp(s - m)
        lse[r] = m + np.log(e.sum())
        o[r] = (e / e.sum()) @ v
    return o, lse


def backward_rows(q, k, v, o, do, lse, causal: bool, scale: float, rows):
    """dQ at the listed query rows and dK, dV at the listed key rows of one head.

    Inputs are one head's [S, D] arrays and its LSE [S] (the O and LSE that the
    backward is fed, like ``backward``).  Each row comes from the definition in
    the module docstring, without forming an S x S matrix:
      dQ_i = scale * sum_j P_ij (dP_ij - delta_i) k_j        (row i of P and dP)
      dK_j = scale * sum_i P_ij (dP_ij - delta_i) q_i        (column j of P and dP)
      dV_j = sum_i P_ij dO_i
    Returns (dQ, dK, dV), each [len(rows), D] fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    S, D = q.shape
    delta = (do * o).sum(axis=1)                    # delta_i for every query row
    dq = np.empty((len(rows), D))
    dk = np.empty((len(rows), D))
    dv = np.empty((len(rows), D))
    for r, i in enumerate(rows):
        # query row i: P_i. and dP_i. over all keys
        s = scale * (k @ q[i])
        if causal:
            s[i + 1:] = -np.inf
        p = np.exp(s - lse[i])
        dp = v @ do[i]
        dq[r] = scale * ((p * (dp - delta[i])) @ k)
        # key row j = i: P_.j and dP_.j over all queries
        j = i
        s = scale * (q @ k[j])
        if causal:
            s[:j] = -np.inf
        p = np.exp(s - lse)
        dp = do @ v[j]
        dk[r] = scale * ((p * (dp - delta)) @ q)
        dv[r] = p @ do
    return dq, dk, dv
