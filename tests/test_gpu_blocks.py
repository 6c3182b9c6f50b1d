"""Thread blocks that take query tiles in turn against one block per tile.

By default one thread block per SM takes 128-row query tiles one after the
other (fat_block_mode): the next tile's Q, first K tiles and first S tiles
overlap the last tile's epilogue, and ring slots and barrier phases run on
from tile to tile.  Each tile goes through the same arithmetic whichever
block runs it, so the two block modes must agree bit for bit (O, LSE and the
count of rows that took the one-row-tile second pass).  Every shape here has
more tiles than the GPU has SMs, so blocks of the default mode run several
tiles, including ragged last tiles, causal tiles of every length and (stress)
tiles whose second pass falls between other tiles.  One test also compares
the default mode with the oracle on whole tensors.
"""
import pytest
import torch

from tensorized_online_softmax_gb300 import inputs as gen

from gpu_helpers import compare, oracle_full, run_cuda, to_dev, tol_key

pytestmark = pytest.mark.gpu

CASES = [
    # (workload, variant, extra binding arguments)
    (gen.WORKLOADS["b4h16n2048d128"], "tensor", {}),
    (gen.WORKLOADS["b4h16n2048d128_causal"], "tensor", {}),
    (gen.WORKLOADS["b4h16n2048d128_causal"], "vec", {}),
    (gen.WORKLOADS["b4h16n2048d128_causal"], "tensor_l", {}),
    (gen.Workload("b2h16n3000d64_causal_x16", 2, 16, 3000, 64, True, 16, seed=7101), "tensor",
     {}),
    (gen.Workload("b2h16n2048d128_causal_x128", 2, 16, 2048, 128, True, 128, seed=7102),
     "tensor", {"z_mode": "tensor"}),
    (gen.Workload("b2h16n2048d64_x128", 2, 16, 2048, 64, False, 128, seed=7103), "tensor_l",
     {"z_mode": "tensor"}),
    (gen.Workload("fp16_b2h16n2048d128_causal", 2, 16, 2048, 128, True, 64, dtype="fp16",
                  seed=7104), "tensor", {}),
    (gen.WORKLOADS["fp8_b4h16n4096d128"], "tensor", {}),
    (gen.WORKLOADS["stress_b1h32n16384d64"], "tensor", {}),
    # a shift of 120 nats: every tile holding a shifted row takes the second pass
    (gen.WORKLOADS["stress_b1h32n16384d64"].with_(name="stress_forced", N=4096,
                                                   shift_coord=31.0), "tensor", {}),
    (gen.WORKLOADS["stress_b1h32n16384d64"].with_(name="stress_forced_x128", N=4096, X=128,
                                                   shift_coord=31.0), "tensor_l", {}),
]


@pytest.mark.parametrize("w,variant,kw", CASES,
                         ids=[f"{c[0].name}-{c[1]}{'-zt' if c[2] else ''}" for c in CASES])
def test_block_modes_agree(cuda_device, w, variant, kw):
    inp = to_dev(gen.make_inputs(w))
    n_tiles = w.B * w.H * ((w.N + 127) // 128)
    assert n_tiles > torch.cuda.get_device_properties(0).multi_processor_count
    res = {}
    for mode in ("auto", "per_tile"):
        fb = torch.zeros(1, dtype=torch.int32, device="cuda")
        o, lse = run_cuda(w, inp, variant, block_mode=mode, fallback_rows=fb, **kw)
        res[mode] = (o, lse, int(fb.item()))
    (o_a, lse_a, fb_a), (o_t, lse_t, fb_t) = res["auto"], res["per_tile"]
    assert torch.equal(o_a, o_t), "O differs between block modes"
    assert torch.equal(lse_a, lse_t), "LSE differs between block modes"
    assert fb_a == fb_t
    if w.shift_coord == 31.0:
        assert fb_a > 0, "the shifted rows should take the second pass"


@pytest.mark.parametrize("variant", ["tensor", "vec"])
@pytest.mark.parametrize("causal", [False, True])
def test_tiles_in_turn_match_oracle(cuda_device, causal, variant):
    # 60 heads x 6 query tiles (the last one ragged): blocks take two or
    # three tiles each
    w = gen.Workload("b1h60n700d64", 1, 60, 700, 64, causal, 64, seed=7105)
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant)
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"tiles in turn {variant} causal={causal}",
            variant=variant)
