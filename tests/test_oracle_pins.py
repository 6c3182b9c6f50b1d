"""Pins for the CPU oracle: checks against things other than the oracle itself.

The oracle computes plain softmax attention, the quantity the fused flow of
"FlashAttention-T: Towards Fully Tensorized Attention by Exploiting
Tensor-Vector Parallelism" (section A3, Fig. 2) produces block by block.  It is
pinned here by
  * hand-worked examples (tests/golden/worked_examples.json),
  * brute force in long double on tiny inputs,
  * closed forms (identical keys, one dominant key, constant V, causal row 0, N=1),
  * invariants (LSE bounds, key/value permutation, logit shift, linearity in V,
    V = identity exposing the probabilities exp(s - LSE)),
  * the surrogate-maximum algorithm of section A2 (Algorithm 1) agreeing with
    the exact-maximum definition, and reporting all-underflow when the gap
    between the surrogate and the exact maximum is beyond the double range,
and a mutation test showing that planted mistakes in the oracle fail these pins.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def _logits(q, k, scale):
    """scale * Q K^T per (b, h) with numpy's matmul (a library primitive)."""
    return scale * np.einsum("bhid,bhjd->bhij", q, k)


# --------------------------------------------------------------------------
# pin suites, each a function of a loaded oracle library (reused by the
# mutation test below)
# --------------------------------------------------------------------------

def _eval_expr(x):
    if isinstance(x, (int, float)):
        return float(x)
    ns = {"e": math.e, "ln": math.log, "ln2": math.log(2), "ln3": math.log(3),
          "ln4": math.log(4), "ln6": math.log(6)}
    return float(eval(x, {"__builtins__": {}}, ns))


def pins_golden(lib):
    cases = json.load(open(GOLDEN))["cases"]
    for case in cases:
        q = np.array([[_eval_expr(x) for x in r] for r in case["q"]])[None, None]
        k = np.array([[_eval_expr(x) for x in r] for r in case["k"]])[None, None]
        v = np.array([[_eval_expr(x) for x in r] for r in case["v"]])[None, None]
        for mode in ("noncausal", "causal"):
            exp_o = np.array([[_eval_expr(x) for x in r] for r in case[mode]["o"]])
            exp_lse = np.array([_eval_expr(x) for x in case[mode]["lse"]])
            o, lse = oracle.attn_fwd(q, k, v, mode == "causal", case["scale"], lib=lib)
            np.testing.assert_allclose(o[0, 0], exp_o, rtol=0, atol=1e-12,
                                       err_msg=f"{case['name']} {mode} O")
            np.testing.assert_allclose(lse[0, 0], exp_lse, rtol=0, atol=1e-12,
                                       err_msg=f"{case['name']} {mode} LSE")


BRUTE_SHAPES = [(1, 1, 1, 1), (1, 2, 7, 3), (2, 1, 16, 8), (1, 1, 64, 16), (2, 3, 33, 5)]


def pins_bruteforce(lib):
    for n, (B, H, N, d) in enumerate(BRUTE_SHAPES):
        q, k, v = (_rand((B, H, N, d), 10 * n + i, std=1.5) for i in range(3))
        scale = 0.3 + 0.1 * n
        for causal in (False, True):
            o, lse = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
            on, lsen = oracle.attn_naive(q, k, v, causal, scale, lib=lib)
            np.testing.assert_allclose(o, on, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lsen, rtol=0, atol=1e-12)


def pins_closed_forms(lib):
    B, H, N, d = 2, 2, 37, 6
    # identical keys: uniform weights -> O_i = mean of the allowed v_j,
    # LSE_i = s + ln |J_i|
    q = _rand((B, H, N, d), 1)
    k = np.broadcast_to(_rand((B, H, 1, d), 2), (B, H, N, d)).copy()
    v = _rand((B, H, N, d), 3)
    scale = 0.7
    s = scale * np.einsum("bhid,bhd->bhi", q, k[:, :, 0])
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
        if causal:
            cnt = np.arange(1, N + 1)
            mean = np.cumsum(v, axis=2) / cnt[None, None, :, None]
        else:
            cnt = np.full(N, N)
            mean = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
        np.testing.assert_allclose(o, mean, atol=1e-12)
        np.testing.assert_allclose(lse, s + np.log(cnt)[None, None], atol=1e-12)
    # one dominant logit: a reserved coordinate gives key j* a +60 lead for every row
    q = _rand((1, 1, N, d), 4, std=0.2)
    k = _rand((1, 1, N, d), 5, std=0.2)
    q[..., -1] = 1.0
    k[..., -1] = 0.0
    jstar = 11
    k[0, 0, jstar, -1] = 60.0
    o, lse = oracle.attn_fwd(q, k, v[:1, :1], False, 1.0, lib=lib)
    # the other keys weigh at most (N - 1) e^-60 ~ 3e-25 together
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, jstar], (N, d)), atol=1e-14)
    # constant V -> O == that constant (any logits, causal or not)
    c = _rand((d,), 6)
    vc = np.broadcast_to(c, (B, H, N, d)).copy()
    qq, kk = _rand((B, H, N, d), 7, 2.0), _rand((B, H, N, d), 8, 2.0)
    for causal in (False, True):
        o, _ = oracle.attn_fwd(qq, kk, vc, causal, 0.5, lib=lib)
        np.testing.assert_allclose(o, vc, atol=1e-12)
    # causal row 0 sees only key 0: O_0 = v_0, LSE_0 = s_00
    o, lse = oracle.attn_fwd(qq, kk, v, True, 0.5, lib=lib)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.5 * np.sum(qq[:, :, 0] * kk[:, :, 0], -1), atol=1e-12)
    # N = 1: O = v, LSE = s
    o, lse = oracle.attn_fwd(qq[:, :, :1], kk[:, :, :1], v[:, :, :1], False, 0.5, lib=lib)
    np.testing.assert_allclose(o, v[:, :, :1], atol=1e-14)
    np.testing.assert_allclose(lse[..., 0], 0.5 * np.sum(qq[:, :, 0] * kk[:, :, 0], -1), atol=1e-12)


def pins_invariants(lib):
    B, H, N, d = 1, 3, 45, 8
    q, k, v = _rand((B, H, N, d), 21, 1.3), _rand((B, H, N, d), 22, 1.3), _rand((B, H, N, d), 23)
    scale = 0.4
    S = _logits(q, k, scale)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        Sm = np.where(np.tril(np.ones((N, N), bool)), S, -np.inf) if causal else S
        m = Sm.max(-1)
        cnt = np.arange(1, N + 1) if causal else np.full(N, N)
        assert np.all(lse >= m - 1e-12)
        assert np.all(lse <= m + np.log(cnt) + 1e-12)
        # doubling V doubles O
        o2, lse2 = oracle.attn_fwd(q, k, 2 * v, causal, scale, lib=lib)
        np.testing.assert_allclose(o2, 2 * o, atol=1e-12)
        np.testing.assert_allclose(lse2, lse, atol=0)
    # joint key/value permutation leaves the non-causal result unchanged
    perm = np.random.default_rng(3).permutation(N)
    o, lse = oracle.attn_fwd(q, k, v, False, scale, lib=lib)
    op, lsep = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], False, scale, lib=lib)
    np.testing.assert_allclose(op, o, atol=1e-12)
    np.testing.assert_allclose(lsep, lse, atol=1e-12)
    # adding delta to every logit of a row (reserved coordinate) keeps O, shifts LSE
    q2, k2 = q.copy(), k.copy()
    q2[..., -1] = 0.0
    k2[..., -1] = 0.0
    o_ref, lse_ref = oracle.attn_fwd(q2, k2, v, True, scale, lib=lib)
    delta = 7.25
    q2[..., -1] = 1.0
    k2[..., -1] = delta / scale
    o_sh, lse_sh = oracle.attn_fwd(q2, k2, v, True, scale, lib=lib)
    np.testing.assert_allclose(o_sh, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse_sh, lse_ref + delta, atol=1e-12)
    # V = identity (d = N): O is the probability matrix, rows sum to 1 and
    # O_ij = exp(s_ij - LSE_i)
    n = 24
    qi, ki = _rand((1, 1, n, n), 31), _rand((1, 1, n, n), 32)
    eye = np.eye(n)[None, None]
    Si = _logits(qi, ki, 0.3)
    for causal in (False, True):
        P, lse = oracle.attn_fwd(qi, ki, eye, causal, 0.3, lib=lib)
        np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-13)
        expect = np.exp(Si - lse[..., None])
        if causal:
            expect = np.where(np.tril(np.ones((n, n), bool)), expect, 0.0)
        np.testing.assert_allclose(P, expect, atol=1e-13)


ALL_PINS = [pins_golden, pins_bruteforce, pins_closed_forms, pins_invariants]


# --------------------------------------------------------------------------
# tests
# --------------------------------------------------------------------------

@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle._get())


def test_row_selection_matches_full():
    q, k, v = (_rand((2, 2, 70, 8), 40 + i) for i in range(3))
    o, lse = oracle.attn_fwd(q, k, v, True, 0.35)
    os_, lses = oracle.attn_fwd(q, k, v, True, 0.35, rows=slice(3, 70, 5))
    np.testing.assert_array_equal(os_[:, :, 3::5], o[:, :, 3::5])
    np.testing.assert_array_equal(lses[:, :, 3::5], lse[:, :, 3::5])
    assert np.isnan(lses[:, :, 4]).all()


@pytest.mark.parametrize("X", [16, 32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_surrogate_max_equals_exact_max(X, causal):
    """Section A2: with m_hat >= m the uniform offset cancels in P~ / l."""
    B, H, N, d = 1, 2, 300, 16  # N not a multiple of any tile: ragged last tile
    q, k, v = _rand((B, H, N, d), 50, 1.5), _rand((B, H, N, d), 51, 1.5), _rand((B, H, N, d), 52)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.25)
    for BN in (128, 64):
        os_, lses, gap, n_under = oracle.attn_surrogate(q, k, v, causal, 0.25, X, 128, BN)
        assert n_under == 0
        assert np.all(gap >= 0)  # m_hat[i] >= m[i]
        np.testing.assert_allclose(os_, o, atol=1e-12)
        np.testing.assert_allclose(lses, lse, atol=1e-12)


def test_surrogate_gap_is_zero_for_one_row_tiles():
    q, k, v = (_rand((1, 1, 64, 8), 60 + i) for i in range(3))
    _, _, gap, _ = oracle.attn_surrogate(q, k, v, False, 0.5, X=1, BM=64, BN=32)
    np.testing.assert_array_equal(gap, 0.0)


def test_surrogate_reports_all_underflow():
    """A row whose X-tile neighbour leads by > 1100 nats underflows entirely in
    double (exp(-745) is the smallest double); the exact definition does not."""
    B, H, N, d = 1, 1, 128, 8
    q, k, v = _rand((B, H, N, d), 70), _rand((B, H, N, d), 71), _rand((B, H, N, d), 72)
    q[..., -1] = 0.0
    k[..., -1] = 0.0
    q[0, 0, 5, -1] = 40.0   # row 5 ...
    k[0, 0, 77, -1] = 30.0  # ... meets key 77 with a +1200 logit
    o_ex, lse_ex = oracle.attn_fwd(q, k, v, False, 1.0)
    assert np.isfinite(o_ex).all() and np.isfinite(lse_ex).all()
    o, lse, gap, n_under = oracle.attn_surrogate(q, k, v, False, 1.0, X=16, BM=128, BN=128)
    # every other row of the 16-row tile holding row 5 underflows
    assert n_under == 15
    tile = np.arange(16)
    assert np.all(gap[0, 0, tile[tile != 5]] > 1100 * math.log2(math.e))
    assert np.isnan(o[0, 0, 0]).all()
    # rows of other tiles are exact
    np.testing.assert_allclose(o[0, 0, 16:], o_ex[0, 0, 16:], atol=1e-12)
    # with one-row tiles (X = 1) the surrogate is the exact maximum: no underflow
    o1, lse1, gap1, n1 = oracle.attn_surrogate(q, k, v, False, 1.0, X=1, BM=128, BN=128)
    assert n1 == 0
    np.testing.assert_allclose(o1, o_ex, atol=1e-12)


# --------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin
# --------------------------------------------------------------------------

MUTANTS = {
    "scale_dropped": ("s[j] = jb->scale * dot;", "s[j] = dot;"),
    "causal_off_by_one": ("long nkeys = jb->causal ? i + 1 + (jb->Nk - jb->Nq) : N;",
                          "long nkeys = jb->causal ? i + (jb->Nk - jb->Nq) : N;"),
    "lse_log2": ("jb->lse[bh * jb->Nq + i] = m + log(l);",
                 "jb->lse[bh * jb->Nq + i] = m + log2(l);"),
    "lse_max_dropped": ("jb->lse[bh * jb->Nq + i] = m + log(l);", "jb->lse[bh * jb->Nq + i] = log(l);"),
    "no_normalisation": ("for (long c = 0; c < d; ++c) oi[c] /= l;", ""),
    "exp_sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "q_k_swapped": ("dot += qi[c] * kj[c];",
                    "dot += jb->k[(bh * N + i) * d + c] * jb->q[(bh * jb->Nq + j) * d + c];"),
    "v_index": ("const double *vj = vb + j * d;", "const double *vj = vb + (N - 1 - j) * d;"),
    "v_transposed": ("for (long c = 0; c < d; ++c) oi[c] += w * vj[c];",
                     "for (long c = 0; c < d; ++c) oi[c] += w * vb[(c % N) * d + (j % d)];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found"
    mpath = tmp_path / "oracle_mut.c"
    mpath.write_text(src.replace(old, new))
    so = str(tmp_path / "liboracle_mut.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", so, str(mpath), "-lm", "-lpthread"], check=True)
    lib = oracle.load(so)
    failures = 0
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(lib)
        except (AssertionError, RuntimeError, ValueError):
            failures += 1
    assert failures >= 1, f"no pin caught the planted mistake {name}"


def test_rectangular_rows_equal_the_tail_of_a_square_problem():
    """Nq queries against Nk keys (causal: the queries are the last Nq key
    positions) give exactly the last Nq rows of the square problem, which is
    itself pinned by brute force above."""
    B, H, N, d = 2, 2, 70, 8
    q, k, v = (_rand((B, H, N, d), 80 + i) for i in range(3))
    for causal in (False, True):
        o_sq, lse_sq = oracle.attn_naive(q, k, v, causal, 0.4)
        for nq in (1, 5, 70):
            o, lse = oracle.attn_fwd_qk(q[:, :, N - nq:], k, v, causal, 0.4)
            np.testing.assert_allclose(o, o_sq[:, :, N - nq:], atol=1e-12)
            np.testing.assert_allclose(lse, lse_sq[:, :, N - nq:], atol=1e-12)


def test_rectangular_non_causal_ignores_key_order_and_rejects_short_causal():
    q = _rand((1, 1, 3, 4), 90)
    k, v = _rand((1, 1, 11, 4), 91), _rand((1, 1, 11, 4), 92)
    perm = np.random.default_rng(4).permutation(11)
    o, lse = oracle.attn_fwd_qk(q, k, v, False, 0.7)
    op, lsep = oracle.attn_fwd_qk(q, k[:, :, perm], v[:, :, perm], False, 0.7)
    np.testing.assert_allclose(op, o, atol=1e-12)
    np.testing.assert_allclose(lsep, lse, atol=1e-12)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd_qk(_rand((1, 1, 12, 4), 93), k, v, True, 0.7)


# --------------------------------------------------------------------------
# negative pin: an update rule that must NOT agree with the oracle
# --------------------------------------------------------------------------

def _blocked_online(q, k, v, scale, block, factor_on_new):
    """Blocked online softmax over key blocks, with the per-row rescale
    factor exp(m_old - m_new) placed on the running output (the correct
    update) or, when ``factor_on_new`` is set, on the new block's term P V
    (the update rule of the first PyTorch example in the FA-T post,
    "FlashAttention-T：张量化注意力机制优化方案", which leaves the old
    output scaled only by l_old / l_new).  The row sum l is carried the same
    way in both.  Returns (O, l); LSE = m + ln l for the correct rule."""
    B, H, N, d = q.shape
    out = np.zeros_like(v)
    l_run = np.zeros((B, H, N, 1))
    m_run = np.full((B, H, N, 1), -np.inf)
    for j in range(0, N, block):
        s = scale * np.einsum("bhid,bhjd->bhij", q, k[:, :, j:j + block])
        m_new = np.maximum(m_run, s.max(axis=-1, keepdims=True))
        alpha = np.exp(m_run - m_new)  # 0 on the first block (m_run = -inf)
        p = np.exp(s - m_new)
        l_new = alpha * l_run + p.sum(axis=-1, keepdims=True)
        pv = np.einsum("bhij,bhjd->bhid", p, v[:, :, j:j + block])
        if factor_on_new:
            out = (l_run / l_new) * out + (alpha / l_new) * pv
        else:
            out = (alpha * l_run / l_new) * out + pv / l_new
        m_run, l_run = m_new, l_new
    return out, m_run[..., 0] + np.log(l_run[..., 0])


def test_misplaced_rescale_rule_disagrees_with_the_oracle():
    """The FA-T post's first example multiplies the new block's P V by
    exp(m_old - m_new) instead of the running output.  On random data that
    rule must disagree with the oracle (so the oracle cannot have adopted
    it), while the same blocked loop with the factor on the running output
    agrees with the oracle, and the oracle agrees with brute force."""
    B, H, N, d, block = 2, 2, 128, 16, 32
    q, k, v = (_rand((B, H, N, d), 300 + i, std=1.2) for i in range(3))
    scale = d ** -0.5
    o, lse = oracle.attn_fwd(q, k, v, False, scale)
    o_bf, lse_bf = oracle.attn_naive(q, k, v, False, scale)
    np.testing.assert_allclose(o, o_bf, atol=1e-12)
    np.testing.assert_allclose(lse, lse_bf, atol=1e-12)
    o_ok, lse_ok = _blocked_online(q, k, v, scale, block, factor_on_new=False)
    np.testing.assert_allclose(o_ok, o, atol=1e-12)
    np.testing.assert_allclose(lse_ok, lse, atol=1e-12)
    o_bad, _ = _blocked_online(q, k, v, scale, block, factor_on_new=True)
    # the first block's contribution is lost (its factor is exp(-inf) = 0)
    # and later ones are mis-weighted: far outside any rounding bar
    assert np.abs(o_bad - o).max() > 0.1
    assert np.abs(o_bad - o).mean() > 1e-2
