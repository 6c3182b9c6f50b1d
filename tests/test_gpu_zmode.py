"""Parity of Z on the tensor pipe (fat_zmode FAT_ZMODE_TENSOR) with the CPU
oracle.

The S MMA adds a bias b = -m_ref / (log2(e) scale), rounded to bf16, through
one more K step against a tile of ones; the vector side folds log2(e) scale b
into the offset of the exponentials.  The attention computed is unchanged, so
the oracle and the accuracy bars are the standard ones.  The growth inputs
change the surrogate maximum on every K/V tile (the bias tiles are rewritten
every time), and the forced-fallback inputs run the second pass, which must
start from zero bias tiles.
"""
import math

import numpy as np
import pytest
import torch

from tensorized_online_softmax_gb300 import inputs as gen

from gpu_helpers import compare, oracle_full, run_cuda, to_dev, tol_key, workload_with_oracle

pytestmark = pytest.mark.gpu

SMALL = [
    # (B, H, N, d, causal); X = 128 throughout
    (1, 2, 256, 128, True),
    (2, 3, 300, 64, True),      # ragged tail
    (1, 1, 7, 128, True),       # shorter than one tile
    (1, 1, 1000, 64, True),
    (2, 2, 640, 128, False),
    (1, 2, 1500, 128, False),   # many tiles, ragged
]


@pytest.mark.parametrize("variant", ["tensor", "tensor_l"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}N{}d{}{}".format(
    s[0], s[1], s[2], s[3], "c" if s[4] else ""))
def test_small_shapes_ztensor(cuda_device, shape, variant):
    B, H, N, d, causal = shape
    w = gen.Workload("small_zt", B, H, N, d, causal, 128, seed=31 + N + d)
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant, z_mode="tensor")
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"z tensor {shape} {variant}",
            variant=variant)


@pytest.mark.parametrize("variant", ["tensor", "tensor_l"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("binades", [3, 20, 120, -20])
def test_growing_maximum_ztensor(cuda_device, binades, causal, variant):
    w = gen.Workload("growth_zt", 1, 2, 1024, 128, causal, 128, kind="growth", seed=4243,
                     growth_nats=binades * math.log(2.0))
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant, z_mode="tensor")
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"z tensor growth {binades} {variant} causal={causal}",
            variant=variant)


def test_fallback_pass_ztensor(cuda_device):
    """A +120-nat logit shift on 1 % of the rows leaves the other rows of
    their 128-row tiles far below the surrogate maximum: those blocks run the
    second (per-row) pass, whose S tiles must carry no bias."""
    w = gen.Workload("stress_zt", 1, 4, 2048, 64, False, 128, kind="stress", seed=99,
                     qk_std=2.8, shift_coord=31.0)
    inp = gen.make_inputs(w)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = run_cuda(w, to_dev(inp), "tensor", z_mode="tensor", fallback_rows=counter)
    assert int(counter.item()) > 0
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what="z tensor fallback")


@pytest.mark.parametrize("variant", ["tensor", "tensor_l"])
def test_full_size_whole_tensor_ztensor(cuda_device, variant):
    """B2 H16 N8192 d128 causal, X = 128, in the launch configuration the
    benchmark times; the whole output against the oracle."""
    w, inp, (o_ref, lse_ref) = workload_with_oracle("b2h16n8192d128_causal")
    o, lse = run_cuda(w, to_dev(inp), variant, z_mode="tensor")
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"z tensor full {variant}", variant=variant)


def test_ztensor_matches_vector_z(cuda_device):
    """Both placements of the subtraction compute the same attention: on the
    same inputs they agree to well within the oracle bars."""
    w = gen.Workload("zt_vs_vz", 2, 4, 2048, 128, True, 128, seed=5150)
    dev = to_dev(gen.make_inputs(w))
    o_v, lse_v = run_cuda(w, dev, "tensor")
    o_t, lse_t = run_cuda(w, dev, "tensor", z_mode="tensor")
    assert (o_v - o_t).abs().max().item() <= 1e-2
    assert (lse_v - lse_t).abs().max().item() <= 5e-4
