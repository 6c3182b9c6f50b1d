"""Pins of the backward-pass oracle to facts other than its own formulas.

* central finite differences of f = sum(O * dO), with O from the C oracle's
  long-double brute force (an independent forward), against dq, dk, dv;
* invariants of softmax attention: moving every key by one vector shifts each
  row's logits by a constant, so the key gradients of a head sum to zero;
  the rows of P sum to one, so the value gradients sum to the sum of dO;
  identical keys make the weights independent of the query, so dq = 0;
* the row-sampled form agrees with the full matrices, and the forward
  quantities it returns agree with the C oracle.
A dropped D term, a wrong sign, a transposed operand or a missing scale each
breaks the finite-difference check; a dropped D also breaks the key-sum one.
"""
import numpy as np
import pytest

import oracle
from oracle.backward import attn_bwd, attn_bwd_sampled

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _f(q, k, v, do, causal, scale):
    o, _ = oracle.attn_naive(q, k, v, causal, scale)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    B, H, N, d = 1, 2, 5, 3
    q, k, v, do = (_rand((B, H, N, d), s) for s in (1, 2, 3, 4))
    scale = 0.7
    dq, dk, dv, _, _ = attn_bwd(q, k, v, do, causal, scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_f(args_p["q"], args_p["k"], args_p["v"], do, causal, scale) -
                        _f(args_m["q"], args_m["k"], args_m["v"], do, causal, scale)) / (2 * h)
        assert np.abs(num - g).max() <= 1e-7 * max(1.0, np.abs(g).max()), name


@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    B, H, N, d = 2, 2, 37, 8
    q, k, v, do = (_rand((B, H, N, d), s) for s in (5, 6, 7, 8))
    dq, dk, dv, _, _ = attn_bwd(q, k, v, do, causal, 0.35)
    assert np.abs(dk.sum(axis=2)).max() <= 1e-11 * np.abs(dk).sum(axis=2).max()
    assert np.abs(dv.sum(axis=2) - do.sum(axis=2)).max() <= 1e-11 * np.abs(do).sum()
    k_same = np.broadcast_to(k[:, :, :1], k.shape).copy()
    dq0, _, _, o, _ = attn_bwd(q, k_same, v, do, causal, 0.35)
    assert np.abs(dq0).max() <= 1e-12
    # identical keys: uniform weights over the allowed keys
    counts = np.arange(1, N + 1)[:, None] if causal else np.full((N, 1), N)
    want = (np.cumsum(v, axis=2) if causal else np.broadcast_to(v.sum(axis=2, keepdims=True),
                                                                 v.shape)) / counts
    assert np.abs(o - want).max() <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_matches_full_and_forward_matches_c_oracle(causal):
    B, H, N, d = 1, 1, 300, 16
    q, k, v, do = (_rand((B, H, N, d), s) for s in (9, 10, 11, 12))
    scale = d ** -0.5
    dq, dk, dv, o, lse = attn_bwd(q, k, v, do, causal, scale)
    o_c, lse_c = oracle.attn_fwd(q, k, v, causal, scale)
    assert np.abs(o - o_c).max() <= 1e-12 and np.abs(lse - lse_c).max() <= 1e-12
    rows = [0, 1, 127, 128, 299]
    sq, sk, sv = attn_bwd_sampled(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, scale, rows, rows)
    for r in rows:
        assert np.abs(sq[r] - dq[0, 0, r]).max() <= 1e-12
        assert np.abs(sk[r] - dk[0, 0, r]).max() <= 1e-12
        assert np.abs(sv[r] - dv[0, 0, r]).max() <= 1e-12
