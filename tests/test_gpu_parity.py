"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every comparison is element by element over whole tensors: small shapes
(several tiles, ragged tails, every X, every variant) and the five full-size
workloads in the launch configuration the benchmark times.  Bars: bf16 O
max-abs <= 2e-2, mean-abs <= 2e-3; e4m3 6e-2 / 6e-3; LSE max-abs <= 1e-3.
They are never widened: an arm that misses one by construction is reported
as an expected failure with its measured error (gpu_helpers.compare).
"""
import numpy as np
import pytest
import torch

import oracle
import tensorized_online_softmax_gb300 as fat
from tensorized_online_softmax_gb300 import inputs as gen

from gpu_helpers import (TOL, compare, error_stats, oracle_full, run_cuda, to_dev, tol_key,
                         workload_with_oracle)

pytestmark = pytest.mark.gpu

VARIANTS = ["tensor", "vec", "tensor_l"]

SMALL = [
    # (B, H, N, d, causal, X)
    (1, 1, 128, 64, False, 16),
    (1, 2, 256, 64, False, 32),
    (1, 2, 256, 128, True, 64),
    (2, 3, 300, 64, True, 64),      # ragged tail, partial second Q tile
    (1, 1, 1, 128, False, 128),     # N = 1
    (1, 1, 7, 64, True, 16),        # shorter than one tile
    (1, 2, 129, 128, False, 64),    # one row past a tile
    (1, 1, 1000, 64, True, 128),
    (2, 2, 640, 128, False, 128),
    (1, 1, 513, 128, True, 32),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}N{}d{}{}X{}".format(
    s[0], s[1], s[2], s[3], "c" if s[4] else "", s[5]))
def test_small_shapes_full_compare(cuda_device, shape, variant):
    B, H, N, d, causal, X = shape
    w = gen.Workload("small", B, H, N, d, causal, X, seed=7 + N + d)
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant)
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"{shape} {variant}",
            variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_workload(cuda_device, variant):
    w = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant)
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"tiny {variant}",
            variant=variant)


FULL = ["b4h16n2048d128", "b4h16n2048d128_causal", "b2h16n8192d128_causal",
        "stress_b1h32n16384d64", "fp8_b4h16n4096d128"]

SMALL_FP8 = [
    # (B, H, N, d, causal, X); e4m3 rows must span 128 bytes, so d = 128
    (1, 2, 256, 128, False, 128),
    (1, 1, 300, 128, True, 64),
    (2, 2, 513, 128, False, 32),
    (1, 1, 77, 128, True, 16),
]


@pytest.mark.parametrize("variant", ["tensor", "vec"])
@pytest.mark.parametrize("shape", SMALL_FP8, ids=lambda s: "B{}H{}N{}d{}{}X{}".format(
    s[0], s[1], s[2], s[3], "c" if s[4] else "", s[5]))
def test_small_shapes_fp8(cuda_device, shape, variant):
    """e4m3 inputs against the e4m3 bars over the whole tensors.

    Causal rows with fewer than 128 allowed keys are the one known exception:
    each of their few weights P~ is stored as e4m3 (3 mantissa bits, relative
    rounding up to 2^-4) before the P V product, and with few terms nothing
    averages out, so such a row's O can be off by up to 2^-4 max|v|.  Every
    other row must meet the bars, and LSE (formed from the unrounded
    weights) must meet 1e-3 everywhere; if the whole tensor then still
    misses the O bars, the case is an expected failure with its measured
    error."""
    B, H, N, d, causal, X = shape
    w = gen.Workload("small_fp8", B, H, N, d, causal, X, dtype="e4m3", seed=17 + N)
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant)
    o_ref, lse_ref = oracle_full(w, inp)
    o_g = o.cpu().double().numpy()
    lse_g = lse.cpu().double().numpy()
    what = f"{shape} {variant}"
    stats = error_stats(o_g, lse_g, o_ref, lse_ref, what)
    assert stats["lse_max"] <= 1e-3, f"{what}: {stats}"
    tol = TOL["e4m3"]
    if stats["o_max"] <= tol["o_max"] and stats["o_mean"] <= tol["o_mean"]:
        return
    keys = np.arange(1, N + 1) if causal else np.full(N, N)
    many = keys >= 128
    assert causal and not many.all(), f"{what}: {stats}"
    if many.any():
        sub = error_stats(o_g[:, :, many], lse_g[:, :, many], o_ref[:, :, many],
                          lse_ref[:, :, many], what)
        assert sub["o_max"] <= tol["o_max"] and sub["o_mean"] <= tol["o_mean"], \
            f"{what} rows with >= 128 keys: {sub}"
    pytest.xfail(f"{what}: e4m3 P~ on causal rows with < 128 keys: measured O max-abs "
                 f"{stats['o_max']:.3g}, mean-abs {stats['o_mean']:.3g} against 6e-2 / 6e-3")


FULL_CASES = [(name, variant) for name in FULL for variant in VARIANTS]


@pytest.mark.parametrize("name,variant", FULL_CASES, ids=[f"{n}-{v}" for n, v in FULL_CASES])
def test_full_size_whole_tensor(cuda_device, name, variant):
    """The five full-size workloads (every head group of the tile order,
    every query and key tile), each variant, O and LSE compared element by
    element with the oracle over the whole output."""
    w, inp, (o_ref, lse_ref) = workload_with_oracle(name)
    o, lse = run_cuda(w, to_dev(inp), variant)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"{name} {variant}", variant=variant)


@pytest.mark.parametrize("X", [32, 128])
def test_identical_keys_give_running_means(cuda_device, X):
    B, H, N, d = 1, 2, 384, 64
    q, k, v = gen.random_qkv(B, H, N, d, seed=3)
    k = k[:, :, :1].expand(B, H, N, d).contiguous()
    for variant in ("tensor", "vec"):
        o, lse = fat.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, X=X, variant=variant)
        mean = torch.cumsum(v.double(), 2) / torch.arange(1, N + 1, dtype=torch.float64)[:, None]
        assert (o.cpu().double() - mean).abs().max() < 2e-2
        s = (q.double() * k[:, :, :1].double()).sum(-1) * d ** -0.5
        want = s + torch.log(torch.arange(1, N + 1, dtype=torch.float64))
        assert (lse.cpu().double() - want).abs().max() < 1e-3


def test_constant_v(cuda_device):
    q, k, v = gen.random_qkv(1, 2, 300, 128, seed=4, std=2.0)
    v = torch.full_like(v, 0.75)
    for variant in ("tensor", "vec"):
        o, _ = fat.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=False, X=128, variant=variant)
        assert (o.cpu() - 0.75).abs().max() < 5e-3


def test_outputs_fully_written_and_deterministic(cuda_device):
    w = gen.Workload("det", 1, 3, 700, 128, True, 64, seed=11)
    inp = to_dev(gen.make_inputs(w))
    o = torch.full((1, 3, 700, 128), float("nan"), device="cuda")
    lse = torch.full((1, 3, 700), float("nan"), device="cuda")
    o1, l1 = fat.attn_fwd(inp["q"], inp["k"], inp["v"], True, w.scale, 64, out=(o, lse))
    torch.cuda.synchronize()
    assert torch.isfinite(o1).all() and torch.isfinite(l1).all()
    o2, l2 = fat.attn_fwd(inp["q"], inp["k"], inp["v"], True, w.scale, 64)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_non_default_stream(cuda_device):
    w = gen.Workload("stream", 1, 2, 256, 64, False, 16, seed=12)
    inp = gen.make_inputs(w)
    dev = to_dev(inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fat.attn_fwd(dev["q"], dev["k"], dev["v"], False, w.scale, 16, stream=s)
    s.synchronize()
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref)


def _stress_forced(shift):
    return gen.Workload("stress_forced", 1, 4, 2048, 64, False, 64, kind="stress", seed=99,
                        qk_std=2.8, shift_coord=shift)


def test_forced_fallback_rows_are_recomputed(cuda_device):
    """A +120-nat shift puts ~173 binades between a tile's surrogate maximum
    and the exact maximum of the unshifted rows: every exponential of those
    rows underflows, the detector flags them and they are recomputed with the
    exact per-row maximum."""
    w = _stress_forced(31.0)
    inp = gen.make_inputs(w)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = run_cuda(w, to_dev(inp), "tensor", fallback_rows=counter)
    assert int(counter.item()) > 0
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what="forced fallback")


def test_default_stress_does_not_fall_back(cuda_device):
    w = _stress_forced(15.5)
    inp = gen.make_inputs(w)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = run_cuda(w, to_dev(inp), "tensor", fallback_rows=counter)
    assert int(counter.item()) == 0
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what="stress 30 nats")


def test_threshold_override_forces_fallback(cuda_device):
    w = _stress_forced(15.5)
    inp = gen.make_inputs(w)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = run_cuda(w, to_dev(inp), "tensor", fallback_rows=counter,
                      underflow_log2_threshold=16.0)
    assert int(counter.item()) > 0
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what="T=16")


def test_bounded_wait_reports_timeout_then_recovers(cuda_device):
    """A poll limit of 1 makes the first wait that is not already satisfied
    give up: the kernel drains what it issued, stops, and the error word
    reports FAT_ERR_DEVICE_TIMEOUT; the next call runs normally."""
    w = gen.Workload("timeout", 1, 2, 1024, 128, False, 64, seed=13)
    inp = gen.make_inputs(w)
    dev = to_dev(inp)
    assert fat.check_device_error() == fat.FAT_OK
    fat.attn_fwd(dev["q"], dev["k"], dev["v"], False, w.scale, 64, wait_poll_limit=1)
    assert fat.check_device_error() == fat.FAT_ERR_DEVICE_TIMEOUT
    assert fat.check_device_error() == fat.FAT_OK
    o, lse = run_cuda(w, dev, "tensor")
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what="after timeout")


def test_bad_arguments_on_device(cuda_device):
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fat.FatError) as e:
        fat.attn_fwd(q, q, q, X=12)
    assert e.value.status == fat.FAT_ERR_INVALID_ARG
    flat = torch.zeros(1 * 1 * 128 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    qm = flat[1:].view(1, 1, 128, 64)
    with pytest.raises(fat.FatError) as e:
        fat.attn_fwd(qm, qm, qm)
    assert e.value.status == fat.FAT_ERR_ALIGNMENT


@pytest.mark.parametrize("variant", ["tensor", "vec"])
def test_phase_trace_is_ordered(cuda_device, variant):
    """The clock stamps of the first thread block follow the pipeline order:
    S received <= m_hat known <= P published (by the softmax set that takes
    the tile) <= MMA issuer saw P <= MMA issuer queued the next work, per K/V
    tile, and the result is unchanged by tracing."""
    w = gen.Workload("trace", 1, 2, 2048, 128, True, 128, seed=21)
    inp = to_dev(gen.make_inputs(w))
    tr = torch.zeros(fat.TRACE_WORDS, dtype=torch.int64, device="cuda")
    o1, l1 = fat.attn_fwd(inp["q"], inp["k"], inp["v"], True, w.scale, 128, variant=variant,
                          trace=tr)
    o2, l2 = fat.attn_fwd(inp["q"], inp["k"], inp["v"], True, w.scale, 128, variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    t = tr.cpu().numpy()
    ev = t[:10 * fat.TRACE_ITERS].reshape(5, 2, fat.TRACE_ITERS)
    n_kv = 2048 // 128  # the first block holds the last 128 query rows
    assert (ev[3, 0, :n_kv] > 0).all() and (ev[3, 0, n_kv:] == 0).all()
    for tt in (0, 1):  # the two softmax sets take alternate K/V tiles
        e = ev[:, tt, tt:n_kv:2]
        assert (e[0] > 0).all() and (ev[0, tt, 1 - tt:n_kv:2] == 0).all()
        assert (e[1] >= e[0]).all() and (e[2] >= e[1]).all()
        assert (np.diff(e[0]) > 0).all()
        # the MMA issuer sees P_j only once its set has published it
        assert (ev[3, 0, tt:n_kv:2] >= e[2]).all()
    assert (ev[4, 0, :n_kv] >= ev[3, 0, :n_kv]).all()
    assert (np.diff(ev[3, 0, :n_kv]) > 0).all()
    assert t[-1] > t[-2] > 0
