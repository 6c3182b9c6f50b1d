"""The host-buffer entry point (fat_attn_fwd_host) streams the problem through
the device in chunks of heads; its results equal those of the device call on
the same inputs bit for bit (the same kernel on the same heads), for ragged
chunkings, and match the oracle."""
import numpy as np
import pytest
import torch

import tensorized_online_softmax_gb300 as fat
from tensorized_online_softmax_gb300 import inputs as gen

from gpu_helpers import compare, oracle_full

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, N, d, causal, X, heads_per_chunk)
    (2, 3, 300, 64, True, 64, 2),     # 6 heads: chunks 2, 2, 2
    (1, 5, 513, 128, False, 128, 2),  # 5 heads: chunks 2, 2, 1 (ragged)
    (2, 4, 1024, 128, True, 128, 0),  # default chunking
    (1, 3, 7, 128, True, 16, 1),      # shorter than one tile, one head per chunk
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}d{}{}X{}hc{}".format(
    c[0], c[1], c[2], c[3], "c" if c[4] else "", c[5], c[6]))
def test_host_entry_equals_device_call(cuda_device, case):
    B, H, N, d, causal, X, hc = case
    w = gen.Workload("host", B, H, N, d, causal, X, seed=808 + N)
    inp = gen.make_inputs(w)
    qh, kh, vh = (inp[n].contiguous().pin_memory() for n in ("q", "k", "v"))
    stream = torch.cuda.Stream()
    o_h, lse_h = fat.attn_fwd_host(qh, kh, vh, causal, w.scale, X, heads_per_chunk=hc,
                                   stream=stream)
    stream.synchronize()
    assert fat.check_device_error() == fat.FAT_OK
    o_d, lse_d = fat.attn_fwd(qh.cuda(), kh.cuda(), vh.cuda(), causal, w.scale, X)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    o_ref, lse_ref = oracle_full(w, inp)
    compare(o_h.numpy(), lse_h.numpy(), o_ref, lse_ref, what=f"host {case}")


def test_host_entry_reuses_workspace_and_outputs(cuda_device):
    """Two calls back to back on one stream with one workspace and one pair
    of output buffers: the second sees its own inputs."""
    w = gen.Workload("host2", 2, 2, 640, 128, False, 128, seed=99)
    a = gen.make_inputs(w)
    b = gen.make_inputs(gen.Workload("host3", 2, 2, 640, 128, False, 128, seed=100))
    nbytes = fat.load_library().fat_attn_fwd_host_workspace_bytes(2, 2, 640, 128, 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = (torch.empty((2, 2, 640, 128), dtype=torch.float32).pin_memory(),
           torch.empty((2, 2, 640), dtype=torch.float32).pin_memory())
    stream = torch.cuda.Stream()
    for inp in (a, b):
        hq, hk, hv = (inp[n].contiguous().pin_memory() for n in ("q", "k", "v"))
        fat.attn_fwd_host(hq, hk, hv, False, w.scale, 128, out=out, workspace=ws,
                          heads_per_chunk=1, stream=stream)
    stream.synchronize()
    o_d, lse_d = fat.attn_fwd(b["q"].cuda(), b["k"].cuda(), b["v"].cuda(), False, w.scale, 128)
    torch.cuda.synchronize()
    assert torch.equal(out[0], o_d.cpu()) and torch.equal(out[1], lse_d.cpu())
