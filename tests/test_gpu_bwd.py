"""Parity of the backward pass (fat_attn_bwd) with the CPU oracle.

P and dS enter their MMAs rounded to bf16 (relative error <= 2^-9) and are
accumulated in fp32, while Q, K, V and dO are exact bf16 inputs.  So with the
exact O and LSE as inputs every gradient element is within 2^-9 (plus fp32
accumulation and ex2.approx, far smaller; 2^-8 is allowed) of the sum of the
absolute values of its products (oracle.backward.attn_bwd_abs_products), and
the tests check that element by element.  With O and LSE from this library's
forward pass (end to end), O's own error enters D = sum dO * O and the bars
are relative to the gradients' size instead.
"""
import numpy as np
import pytest
import torch

import tensorized_online_softmax_gb300 as fat
from oracle.backward import attn_bwd, attn_bwd_abs_products, attn_bwd_sampled
from tensorized_online_softmax_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

SMALL = [
    # (B, H, N, d, causal)
    (1, 2, 128, 64, False),
    (1, 1, 7, 128, True),       # shorter than one tile
    (2, 3, 300, 64, True),      # ragged tail
    (1, 2, 640, 128, False),
    (1, 1, 1000, 128, True),
    (2, 2, 513, 64, False),
]


def _inputs(B, H, N, d, seed):
    q, k, v = gen.random_qkv(B, H, N, d, seed)
    do, _, _ = gen.random_qkv(B, H, N, d, seed + 1)
    return q, k, v, do


def _f64(t):
    return t.double().cpu().numpy()


def _check_elementwise(got, want, bound, what):
    err = np.abs(_f64(got) - want)
    lim = 2.0 ** -8 * bound + 1e-6 * max(1.0, np.abs(want).max())
    worst = float((err / lim).max())
    assert worst <= 1.0, f"{what}: error reaches {worst:.2f} of the bound"
    return worst


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}N{}d{}{}".format(
    s[0], s[1], s[2], s[3], "c" if s[4] else ""))
def test_small_shapes_bwd(cuda_device, shape):
    B, H, N, d, causal = shape
    q, k, v, do = _inputs(B, H, N, d, seed=700 + N + d)
    scale = d ** -0.5
    dq_r, dk_r, dv_r, o_r, lse_r = attn_bwd(_f64(q), _f64(k), _f64(v), _f64(do), causal, scale)
    bq, bk, bv = attn_bwd_abs_products(_f64(q), _f64(k), _f64(v), _f64(do), causal, scale)
    o = torch.from_numpy(o_r).float().cuda()
    lse = torch.from_numpy(lse_r).float().cuda()
    dq, dk, dv = fat.attn_bwd(q.cuda(), k.cuda(), v.cuda(), o, lse, do.cuda(), causal, scale)
    torch.cuda.synchronize()
    assert fat.check_device_error() == fat.FAT_OK
    for name, got, want, bound in (("dq", dq, dq_r, bq), ("dk", dk, dk_r, bk),
                                   ("dv", dv, dv_r, bv)):
        _check_elementwise(got, want, bound, f"{shape} {name}")


@pytest.mark.parametrize("variant", ["tensor", "vec"])
@pytest.mark.parametrize("causal", [False, True])
def test_end_to_end_with_forward(cuda_device, causal, variant):
    """O and LSE from the forward kernel feed the backward kernel."""
    B, H, N, d = 2, 3, 777, 128
    q, k, v, do = _inputs(B, H, N, d, seed=9001)
    scale = d ** -0.5
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = fat.attn_fwd(qc, kc, vc, causal, scale, 128, variant=variant)
    dq, dk, dv = fat.attn_bwd(qc, kc, vc, o, lse, doc, causal, scale)
    torch.cuda.synchronize()
    ref = attn_bwd(_f64(q), _f64(k), _f64(v), _f64(do), causal, scale)[:3]
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        err = np.abs(_f64(got) - want)
        assert err.max() <= 2e-2 * np.abs(want).max(), (name, err.max(), np.abs(want).max())
        assert err.mean() <= 5e-3 * np.abs(want).mean(), (name, err.mean(), np.abs(want).mean())


def _forward_f64(qc, kc, vc, causal, scale):
    """O and LSE in float64 on the device (plain PyTorch, one head at a time):
    inputs for the backward kernel accurate far beyond the bars below."""
    B, H, N, d = qc.shape
    o = torch.empty((B, H, N, d), dtype=torch.float32, device=qc.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=qc.device)
    for b in range(B):
        for h in range(H):
            s_ = (qc[b, h].double() @ kc[b, h].double().T) * scale
            if causal:
                s_.masked_fill_(torch.ones(N, N, dtype=torch.bool, device=qc.device).triu(1),
                                float("-inf"))
            l_ = torch.logsumexp(s_, dim=1)
            o[b, h] = (torch.exp(s_ - l_[:, None]) @ vc[b, h].double()).float()
            lse[b, h] = l_.float()
            del s_
    return o, lse


@pytest.mark.parametrize("shape", [(2, 16, 8192, 128, True), (4, 16, 2048, 128, False),
                                   (1, 32, 16384, 64, False)],
                         ids=["b2h16n8192d128c", "b4h16n2048d128", "b1h32n16384d64"])
def test_full_size_sampled_bwd(cuda_device, shape):
    """Shapes of the forward workloads, in the launch configuration of the
    benchmark; the oracle gives dq at sampled query rows and dk, dv at sampled
    key rows of two heads."""
    B, H, N, d, causal = shape
    q, k, v, do = _inputs(B, H, N, d, seed=31337 + N)
    scale = d ** -0.5
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = _forward_f64(qc, kc, vc, causal, scale)
    dq, dk, dv = fat.attn_bwd(qc, kc, vc, o, lse, doc, causal, scale)
    torch.cuda.synchronize()
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    rows = sorted({0, 1, 127, 128, N // 2, N - 129, N - 1} |
                  set(np.random.default_rng(N).choice(N, 5, replace=False).tolist()))
    for (b, h) in [(0, 0), (B - 1, H - 1)]:
        sq, sk, sv = attn_bwd_sampled(_f64(q[b, h]), _f64(k[b, h]), _f64(v[b, h]),
                                      _f64(do[b, h]), causal, scale, rows, rows)
        for name, got, ref in (("dq", dq, sq), ("dk", dk, sk), ("dv", dv, sv)):
            g = np.stack([_f64(got[b, h, r]) for r in rows])
            w = np.stack([ref[r] for r in rows])
            err = np.abs(g - w)
            assert err.max() <= 1e-2 * np.abs(w).max(), (shape, name, err.max(), np.abs(w).max())
            assert err.mean() <= 4e-3 * np.abs(w).mean(), (shape, name, err.mean(),
                                                          np.abs(w).mean())


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_full_size_whole_tensor_bwd_b4h16n2048(cuda_device, causal):
    """The B4 H16 N2048 d128 benchmark shape (64 heads, 16 key blocks each, the
    launch the benchmark times): every element of dq, dk and dv against the
    oracle, with the oracle's own O and LSE as the forward's outputs, at the
    full-size bars of the sampled test."""
    B, H, N, d = 4, 16, 2048, 128
    q, k, v, do = _inputs(B, H, N, d, seed=4242 + int(causal))
    scale = d ** -0.5
    dq_r, dk_r, dv_r, o_r, lse_r = attn_bwd(_f64(q), _f64(k), _f64(v), _f64(do), causal, scale)
    o = torch.from_numpy(o_r).float().cuda()
    lse = torch.from_numpy(lse_r).float().cuda()
    dq, dk, dv = fat.attn_bwd(q.cuda(), k.cuda(), v.cuda(), o, lse, do.cuda(), causal, scale)
    torch.cuda.synchronize()
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        err = np.abs(_f64(got) - ref)
        assert np.isfinite(err).all(), name
        assert err.max() <= 1e-2 * np.abs(ref).max(), (name, err.max(), np.abs(ref).max())
        assert err.mean() <= 4e-3 * np.abs(ref).mean(), (name, err.mean(), np.abs(ref).mean())


def test_bwd_argument_errors(cuda_device):
    q, k, v, do = (t.cuda() for t in _inputs(1, 1, 256, 64, seed=5))
    o, lse = fat.attn_fwd(q, k, v, False, 0.125, 64)
    with pytest.raises(ValueError):
        fat.attn_bwd(q, k, v, o, lse, do.float(), False, 0.125)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fat.FatError):
        fat.attn_bwd(q, k, v, o, lse, do, False, 0.125, workspace=ws)
