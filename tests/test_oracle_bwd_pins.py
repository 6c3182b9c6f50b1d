"""Pins of the backward-pass oracle to facts other than its own formulas.

* central finite differences of f = sum(O * dO), with O from the C oracle's
  long-double brute force (an independent forward), against dq, dk, dv;
* invariants of softmax attention: moving every key by one vector shifts each
  row's logits by a constant, so the key gradients of a head sum to zero;
  the rows of P sum to one, so the value gradients sum to the sum of dO;
  identical keys make the weights independent of the query, so dq = 0;
* the row-sampled form agrees with the full matrices, and the forward
  quantities it returns agree with the C oracle.
A mutation test plants mistakes (a dropped D term, a wrong sign of D, a
missing scale, a transposed operand, P instead of P^T) into a copy of the
oracle and checks that each fails at least one pin.
"""
import importlib.util

import numpy as np
import pytest

import oracle
import oracle.backward as backward

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _f(q, k, v, do, causal, scale):
    o, _ = oracle.attn_naive(q, k, v, causal, scale)
    return float((o * do).sum())


def _check_finite_differences(mod, causal):
    B, H, N, d = 1, 2, 5, 3
    q, k, v, do = (_rand((B, H, N, d), s) for s in (1, 2, 3, 4))
    scale = 0.7
    dq, dk, dv, _, _ = mod.attn_bwd(q, k, v, do, causal, scale)
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


def _check_invariants(mod, causal):
    B, H, N, d = 2, 2, 37, 8
    q, k, v, do = (_rand((B, H, N, d), s) for s in (5, 6, 7, 8))
    dq, dk, dv, _, _ = mod.attn_bwd(q, k, v, do, causal, 0.35)
    assert np.abs(dk.sum(axis=2)).max() <= 1e-11 * np.abs(dk).sum(axis=2).max()
    assert np.abs(dv.sum(axis=2) - do.sum(axis=2)).max() <= 1e-11 * np.abs(do).sum()
    k_same = np.broadcast_to(k[:, :, :1], k.shape).copy()
    dq0, _, _, o, _ = mod.attn_bwd(q, k_same, v, do, causal, 0.35)
    assert np.abs(dq0).max() <= 1e-12
    # identical keys: uniform weights over the allowed keys
    counts = np.arange(1, N + 1)[:, None] if causal else np.full((N, 1), N)
    want = (np.cumsum(v, axis=2) if causal else np.broadcast_to(v.sum(axis=2, keepdims=True),
                                                                 v.shape)) / counts
    assert np.abs(o - want).max() <= 1e-12


def _check_sampled_and_forward(mod, causal):
    B, H, N, d = 1, 1, 300, 16
    q, k, v, do = (_rand((B, H, N, d), s) for s in (9, 10, 11, 12))
    scale = d ** -0.5
    dq, dk, dv, o, lse = mod.attn_bwd(q, k, v, do, causal, scale)
    o_c, lse_c = oracle.attn_fwd(q, k, v, causal, scale)
    assert np.abs(o - o_c).max() <= 1e-12 and np.abs(lse - lse_c).max() <= 1e-12
    rows = [0, 1, 127, 128, 299]
    sq, sk, sv = mod.attn_bwd_sampled(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, scale, rows,
                                      rows)
    for r in rows:
        assert np.abs(sq[r] - dq[0, 0, r]).max() <= 1e-12
        assert np.abs(sk[r] - dk[0, 0, r]).max() <= 1e-12
        assert np.abs(sv[r] - dv[0, 0, r]).max() <= 1e-12


CHECKS = (_check_finite_differences, _check_invariants, _check_sampled_and_forward)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__[len("_check_"):])
def test_pins(check, causal):
    check(backward, causal)


# planted mistakes: each must fail at least one pin
MUTANTS = {
    "dropped_D": ("ds = p * (dp - D[:, None])", "ds = p * dp"),
    "D_sign": ("ds = p * (dp - D[:, None])", "ds = p * (dp + D[:, None])"),
    "dq_scale": ("dq[b, h] = scale * (ds @ k[b, h])", "dq[b, h] = (ds @ k[b, h])"),
    "dk_transposed": ("dk[b, h] = scale * (ds.T @ q[b, h])", "dk[b, h] = scale * (ds @ q[b, h])"),
    "dv_not_transposed": ("dv[b, h] = p.T @ do[b, h]", "dv[b, h] = p @ do[b, h]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(backward.__file__).read()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    path = tmp_path / "backward_mut.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("backward_mut", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    failures = 0
    for check in CHECKS:
        for causal in (False, True):
            try:
                check(mod, causal)
            except AssertionError:
                failures += 1
    assert failures >= 1, f"no pin caught the planted mistake {name}"
