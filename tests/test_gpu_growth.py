"""Parity when the running maximum grows from one K/V tile to the next.

The surrogate maximum of an X-row tile is settled before its exponentials,
and O takes the factor 2^(m_old - m_new) on the vector side whenever it grew.
These inputs raise every row's logits by a fixed amount per 128-key tile, so
each K/V tile after the first raises it: by a few binades, by 20, and by more
than 100 (each tile's terms then leave the earlier ones far out of range).  A
shrinking sequence (the first tile dominates) never raises it.
"""
import math

import pytest

from tensorized_online_softmax_gb300 import inputs as gen

from gpu_helpers import compare, oracle_full, run_cuda, to_dev, tol_key

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", ["tensor", "tensor_l", "vec"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("binades", [3, 20, 120, 140, -20])
def test_growing_maximum(cuda_device, binades, causal, variant):
    w = gen.Workload("growth", 1, 2, 1024, 128, causal, 128, kind="growth", seed=4242,
                     growth_nats=binades * math.log(2.0))
    inp = gen.make_inputs(w)
    o, lse = run_cuda(w, to_dev(inp), variant)
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tol_key(w),
            what=f"growth {binades} binades/tile {variant} causal={causal}",
            variant=variant)
