"""Parity of the fp16-input path (the FA-T summary's FP16-FP32 setting, A4)
with the CPU oracle.

fp16 P~ is formed as 2^(Z + 15) so that its terms use the format's range
(fp16's smallest normal is 2^-14); the default underflow threshold is then
29 binades, and rows beyond it go through the one-row-tile fallback pass.
"""
import numpy as np
import pytest
import torch

from tensorized_online_softmax_gb300 import inputs as gen

from gpu_helpers import compare, oracle_full, run_cuda, to_dev, tol_key

pytestmark = pytest.mark.gpu

SMALL = [
    # (B, H, N, d, causal, X)
    (1, 1, 128, 64, False, 16),
    (1, 2, 256, 128, True, 64),
    (2, 3, 300, 64, True, 64),      # ragged tail
    (1, 1, 7, 64, True, 16),        # shorter than one tile
    (1, 1, 1000, 64, True, 128),
    (2, 2, 640, 128, False, 128),
    (1, 1, 513, 128, True, 32),
]


@pytest.mark.parametrize("variant", ["tensor", "vec", "tensor_l"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}N{}d{}{}X{}".format(
    s[0], s[1], s[2], s[3], "c" if s[4] else "", s[5]))
def test_small_shapes_fp16(cuda_device, shape, variant):
    B, H, N, d, causal, X = shape
    w = gen.Workload("small_fp16", B, H, N, d, causal, X, dtype="fp16", seed=11 + N + d)
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant)
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"fp16 {shape} {variant}",
            variant=variant)


@pytest.mark.parametrize("variant", ["tensor", "vec"])
@pytest.mark.parametrize("shape", [(4, 16, 2048, 128, True, 128), (8, 32, 1024, 64, False, 128)],
                         ids=["b4h16n2048d128c", "b8h32n1024d64"])
def test_full_size_fp16_whole_tensor(cuda_device, shape, variant):
    """Shapes of the pages' sweep (16384 tokens, hidden 2048), whole tensors."""
    B, H, N, d, causal, X = shape
    w = gen.Workload("sweep_fp16", B, H, N, d, causal, X, dtype="fp16", seed=2024 + N)
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant)
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "fp16",
            what=f"fp16 {shape} {variant}", variant=variant)


def test_fp16_stress_falls_back_and_matches(cuda_device):
    """+30 nats on 1% of the rows: unshifted rows that share an X-row tile
    with a shifted one sit 43 binades under the surrogate, past fp16's
    29-binade threshold; they are recomputed with one-row tiles."""
    w = gen.Workload("stress_fp16", 1, 4, 2048, 64, False, 64, dtype="fp16", kind="stress",
                     seed=99, qk_std=2.8, shift_coord=15.5)
    inp = gen.make_inputs(w)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = run_cuda(w, to_dev(inp), "tensor", fallback_rows=counter)
    assert int(counter.item()) > 0
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "fp16", what="fp16 stress")
