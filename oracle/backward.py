"""CPU oracle of the attention backward pass (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this module.

The backward pass recomputes the attention weights from the forward inputs
(the v1 recap of "FlashAttention-T 完全张量化内核与内存布局优化深度剖析",
section "从融合到张量化：FlashAttention 演进脉络": the backward pass keeps only
the output and the softmax statistics and recomputes the rest).  What it
computes is the gradient of the forward pass's plain definition
O = softmax(scale Q K^T [+ causal mask]) V with respect to Q, K and V, for an
upstream gradient dO, written out by the chain rule:

    P    = exp(S - LSE)            S = scale Q K^T, masked keys j > i (causal)
    dV   = P^T dO
    dP   = dO V^T
    D_i  = sum_d dO_id O_id        (= sum_j P_ij dP_ij)
    dS   = P * (dP - D)            (softmax Jacobian, row by row)
    dQ   = scale dS K
    dK   = scale dS^T Q

Everything is float64 numpy, [B, H, N, d]; one head at a time, with matmul
as the only library step.  ``attn_bwd_sampled`` gives the same quantities for
chosen query rows (dQ) and key rows (dK, dV) of one head without forming the
N x N matrices, for sizes where the full matrices would not fit.
"""
from __future__ import annotations

import numpy as np


def _head_probs(q, k, causal: bool, scale: float):
    """P and LSE of one head: q [N, d], k [N, d] -> P [N, N], LSE [N]."""
    s = scale * (q @ k.T)
    if causal:
        n = s.shape[0]
        s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    lse = m[:, 0] + np.log(e.sum(axis=1))
    return np.exp(s - lse[:, None]), lse


def attn_bwd(q, k, v, do, causal: bool, scale: float):
    """Gradients (dq, dk, dv) of sum(O * do) for O = attention(q, k, v).

    Also returns O and LSE (natural log, scaled-logit units) of the forward.
    """
    q, k, v, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, do))
    B, H, N, d = q.shape
    dq, dk, dv, o = (np.zeros_like(q) for _ in range(4))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            p, lse[b, h] = _head_probs(q[b, h], k[b, h], causal, scale)
            o[b, h] = p @ v[b, h]
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            D = (do[b, h] * o[b, h]).sum(axis=1)
            ds = p * (dp - D[:, None])
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv, o, lse


def _head_stats(q, k, v, do, causal: bool, scale: float, block: int = 512):
    """LSE [N] and D [N] of one head, formed in row blocks of the forward."""
    N = q.shape[0]
    lse = np.empty(N)
    D = np.empty(N)
    for r0 in range(0, N, block):
        r1 = min(N, r0 + block)
        s = scale * (q[r0:r1] @ k.T)
        if causal:
            s = np.where(np.arange(N)[None, :] <= np.arange(r0, r1)[:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1)
        lse[r0:r1] = m[:, 0] + np.log(den)
        o = (e @ v) / den[:, None]
        D[r0:r1] = (do[r0:r1] * o).sum(axis=1)
    return lse, D


def attn_bwd_sampled(q, k, v, do, causal: bool, scale: float, qrows, krows):
    """One head ([N, d] arrays): dq at query rows ``qrows`` and dk, dv at key
    rows ``krows``, by the same formulas taken one row or column at a time."""
    q, k, v, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, do))
    N = q.shape[0]
    lse, D = _head_stats(q, k, v, do, causal, scale)
    dq = {}
    for i in qrows:
        s = scale * (k @ q[i])
        keep = np.arange(N) <= i if causal else np.ones(N, dtype=bool)
        p = np.where(keep, np.exp(np.where(keep, s, 0.0) - lse[i]), 0.0)
        ds = p * (v @ do[i] - D[i])
        dq[i] = scale * (ds @ k)
    dk, dv = {}, {}
    for j in krows:
        s = scale * (q @ k[j])
        keep = np.arange(N) >= j if causal else np.ones(N, dtype=bool)
        p = np.where(keep, np.exp(np.where(keep, s, 0.0) - lse), 0.0)
        dv[j] = p @ do
        ds = p * (do @ v[j] - D)
        dk[j] = scale * (ds @ q)
    return dq, dk, dv


def attn_bwd_abs_products(q, k, v, do, causal: bool, scale: float):
    """For each gradient element, the sum of the absolute values of the
    products that form it: (scale |dS| |K|, scale |dS|^T |Q|, P^T |dO|) for
    (dq, dk, dv).

    A gradient formed from operands one of which carries a relative rounding
    error of at most e per entry is within e times this sum of the exact
    gradient (the bound the GPU parity tests apply for bf16 P and dS)."""
    q, k, v, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, do))
    B, H, N, d = q.shape
    bq, bk, bv = (np.zeros_like(q) for _ in range(3))
    for b in range(B):
        for h in range(H):
            p, _ = _head_probs(q[b, h], k[b, h], causal, scale)
            o = p @ v[b, h]
            dp = do[b, h] @ v[b, h].T
            D = (do[b, h] * o).sum(axis=1)
            ads = np.abs(p * (dp - D[:, None]))
            bq[b, h] = scale * (ads @ np.abs(k[b, h]))
            bk[b, h] = scale * (ads.T @ np.abs(q[b, h]))
            bv[b, h] = p.T @ np.abs(do[b, h])
    return bq, bk, bv
