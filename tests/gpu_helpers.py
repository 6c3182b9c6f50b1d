"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs (whole tensors or sampled rows), and
compare with the accuracy bars of the fused-attention forward pass."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tensorized_online_softmax_gb300 as fat
from tensorized_online_softmax_gb300 import inputs as gen

# acceptance bars (max-abs / mean-abs on O, max-abs on LSE); fp16 inputs
# (10-bit mantissa) keep the bf16 bars
TOL = {
    "bf16": dict(o_max=2e-2, o_mean=2e-3, lse_max=1e-3),
    "fp16": dict(o_max=2e-2, o_mean=2e-3, lse_max=1e-3),
    "e4m3": dict(o_max=6e-2, o_mean=6e-3, lse_max=1e-3),
}

# test-side variant names -> (binding variant, l_mode)
VARIANT_ARGS = {"tensor": ("tensor", "vector"), "vec": ("vec", "vector"),
                "tensor_l": ("tensor", "tensor")}


def tol_key(w, variant=None):
    return w.dtype


def lse_xfail_reason(dtype, lse_err):
    """Why the row sum on the tensor pipe may miss the LSE bar (row-sum
    option only).  There l is the sum of the rounded P~ that the P V product
    uses: each term carries a relative rounding of up to 2^-9 (bf16 P~) or
    2^-4 (e4m3 P~), so when a few comparable terms carry a row, or many
    equal terms round the same way, ln l can be off by up to ln(1 + 2^-9) =
    1.95e-3 (bf16) or ln(1 + 2^-4) = 6.1e-2 (e4m3): above the 1e-3 bar.
    (fp16 P~: 2^-11, ln(1 + 2^-11) = 4.9e-4, inside it.)"""
    bound = {"bf16": "ln(1+2^-9) = 1.95e-3", "e4m3": "ln(1+2^-4) = 6.1e-2"}.get(dtype)
    if bound is None:
        return None
    return (f"row sum on the tensor pipe, {dtype} P~: measured LSE max error {lse_err:.3g} "
            f"> 1e-3 (rounding bound {bound})")


def to_dev(inputs, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) and k in ("q", "k", "v") else v)
            for k, v in inputs.items()}


def run_cuda(w: gen.Workload, dev_inputs, variant="tensor", **kw):
    q, k, v = dev_inputs["q"], dev_inputs["k"], dev_inputs["v"]
    var, l_mode = VARIANT_ARGS[variant]
    if w.dtype == "e4m3":
        kw = dict(kw, dtype="e4m3", descales=(dev_inputs["q_descale"], dev_inputs["k_descale"],
                                              dev_inputs["v_descale"]))
    elif w.dtype == "fp16":
        kw = dict(kw, dtype="fp16")
    o, lse = fat.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, X=w.X, variant=var,
                          l_mode=l_mode, **kw)
    torch.cuda.synchronize()
    return o, lse


def oracle_full(w: gen.Workload, inputs):
    return oracle.attn_fwd(gen.widened(inputs, "q"), gen.widened(inputs, "k"),
                           gen.widened(inputs, "v"), w.causal, w.scale)


def sample_rows(N: int, n_random: int, seed: int):
    """Rows on tile edges (0, 127, 128, 255, 256, N-1) plus random rows."""
    rng = np.random.default_rng(seed)
    fixed = [r for r in (0, 1, 127, 128, 255, 256, 383, N // 2, N - 2, N - 1) if 0 <= r < N]
    rnd = rng.choice(N, size=min(n_random, N), replace=False).tolist()
    return sorted(set(fixed + rnd))


def oracle_sampled(w: gen.Workload, inputs, heads, rows):
    """Oracle O/LSE for the given (b, h) heads and query rows only."""
    out = {}
    q64 = gen.widened(inputs, "q")
    k64 = gen.widened(inputs, "k")
    v64 = gen.widened(inputs, "v")
    for (b, h) in heads:
        qs = q64[b:b + 1, h:h + 1].numpy()
        ks = k64[b:b + 1, h:h + 1].numpy()
        vs = v64[b:b + 1, h:h + 1].numpy()
        for r in rows:
            o, lse = oracle.attn_fwd(qs, ks, vs, w.causal, w.scale, rows=slice(r, r + 1))
            out[(b, h, r)] = (o[0, 0, r], lse[0, 0, r])
    return out


def error_stats(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Max-abs / mean-abs error of O and max-abs error of LSE, element by
    element in float64 (in slices of rows, so whole full-size tensors fit)."""
    o_gpu = np.asarray(o_gpu)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert np.isfinite(lse_gpu).all(), f"{what}: non-finite LSE"
    d = o_gpu.shape[-1]
    og = o_gpu.reshape(-1, d)
    orf = np.asarray(o_ref).reshape(-1, d)
    o_max, o_sum = 0.0, 0.0
    step = max(1, (1 << 22) // d)
    for r0 in range(0, og.shape[0], step):
        g = og[r0:r0 + step].astype(np.float64)
        assert np.isfinite(g).all(), f"{what}: non-finite O"
        e = np.abs(g - orf[r0:r0 + step])
        o_max = max(o_max, float(e.max()))
        o_sum += float(e.sum())
    lerr = np.abs(lse_gpu - lse_ref)
    return dict(o_max=o_max, o_mean=o_sum / max(1, og.size), lse_max=float(lerr.max()))


_ORACLE_CACHE: dict = {}


def workload_with_oracle(name: str):
    """(workload, host inputs, (O, LSE) of the oracle) for a named workload,
    keeping only the latest one (full-size oracle results are large)."""
    if name not in _ORACLE_CACHE:
        _ORACLE_CACHE.clear()
        w = gen.WORKLOADS[name]
        inp = gen.make_inputs(w)
        _ORACLE_CACHE[name] = (w, inp, oracle_full(w, inp))
    return _ORACLE_CACHE[name]


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype="bf16", what="", variant=None):
    """Element-by-element comparison against the bars; returns the error stats.

    The bars are never widened.  One arm is known to miss the LSE bar by
    construction: the row sum on the tensor pipe (``variant="tensor_l"``)
    with bf16 or e4m3 P~ (see :func:`lse_xfail_reason`).  It must still meet
    the O bars; when its LSE error is above 1e-3 the test is reported as an
    expected failure with the measured error, never as a pass.
    """
    tol = TOL[dtype]
    stats = error_stats(o_gpu, lse_gpu, o_ref, lse_ref, what)
    assert stats["o_max"] <= tol["o_max"], f"{what}: {stats}"
    assert stats["o_mean"] <= tol["o_mean"], f"{what}: {stats}"
    if stats["lse_max"] > tol["lse_max"] and variant == "tensor_l":
        reason = lse_xfail_reason(dtype, stats["lse_max"])
        if reason is not None:
            import pytest
            pytest.xfail(f"{what}: {reason}")
    assert stats["lse_max"] <= tol["lse_max"], f"{what}: {stats}"
    return stats


def compare_sampled(o_gpu, lse_gpu, ref: dict, dtype="bf16", what="", variant=None):
    keys = sorted(ref)
    og = np.stack([o_gpu[b, h, r].double().cpu().numpy() for (b, h, r) in keys])
    lg = np.array([float(lse_gpu[b, h, r]) for (b, h, r) in keys])
    orf = np.stack([ref[key][0] for key in keys])
    lrf = np.array([ref[key][1] for key in keys])
    return compare(og, lg, orf, lrf, dtype, what, variant)
