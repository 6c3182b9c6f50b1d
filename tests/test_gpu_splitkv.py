"""Split-KV forward (Nq query rows against Nk keys, the key range split
across thread blocks, partial results merged by LSE weights) against the
oracle of the same rectangular problem.  Bars: bf16 O max-abs <= 2e-2,
mean-abs <= 2e-3, LSE max-abs <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import tensorized_online_softmax_gb300 as fat

from gpu_helpers import compare

pytestmark = pytest.mark.gpu


def _inputs(B, H, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    return q, k, v


CASES = [
    # (B, H, Nq, Nk, d, causal, splits)
    (2, 4, 1, 8192, 128, False, None),   # decode, one query per head
    (2, 4, 1, 8192, 128, False, 64),
    (1, 8, 16, 4096, 128, True, 7),      # speculative tokens at the end of the sequence
    (2, 2, 128, 3000, 64, True, 5),      # ragged key count
    (1, 2, 300, 5000, 128, False, 3),    # two query blocks, ragged rows
    (1, 2, 2048, 2048, 128, True, 8),    # early query blocks get empty key ranges
    (1, 1, 200, 200, 128, True, 1),      # a single range: direct outputs
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}d{}{}s{}".format(
    c[0], c[1], c[2], c[3], c[4], "c" if c[5] else "", c[6]))
def test_splitkv_matches_oracle(cuda_device, case):
    B, H, Nq, Nk, d, causal, splits = case
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=Nq + Nk + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = fat.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal, scale, 128, splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attn_fwd_qk(q.double(), k.double(), v.double(), causal, scale)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what=str(case))


def test_split_count_does_not_change_the_result_beyond_rounding(cuda_device):
    q, k, v = (t.cuda() for t in _inputs(1, 4, 64, 6000, 128, seed=5))
    o1, l1 = fat.attn_fwd_splitkv(q, k, v, False, None, 128, 1)
    for s in (2, 9, 47):
        o2, l2 = fat.attn_fwd_splitkv(q, k, v, False, None, 128, s)
        torch.cuda.synchronize()
        assert (o1 - o2).abs().max().item() < 2e-3
        assert (l1 - l2).abs().max().item() < 1e-4


def test_square_splitkv_equals_the_fused_path(cuda_device):
    q, k, v = (t.cuda() for t in _inputs(2, 2, 1024, 1024, 128, seed=6))
    o1, l1 = fat.attn_fwd(q, k, v, True, None, 128)
    o2, l2 = fat.attn_fwd_splitkv(q, k, v, True, None, 128, 1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
