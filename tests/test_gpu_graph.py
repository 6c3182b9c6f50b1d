"""The forward and backward calls captured in a CUDA graph.

A caller that replays a training or serving step as a CUDA graph captures our
calls on its stream: the forward kernel, and for the backward the
preparation kernel followed by the fused kernel (at d = 128 launched with
programmatic stream serialisation, which capture turns into a programmatic
edge of the graph).  Replays must give what eager calls give, and must read
the graph's input buffers as they are at replay time.  The first call on a
device sets up per-device state, so eager calls come before the capture.
"""
import pytest
import torch

import tensorized_online_softmax_gb300 as fat
from tensorized_online_softmax_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def _eager(q, k, v, do, causal, scale, X):
    o, lse = fat.attn_fwd(q, k, v, causal, scale, X)
    dq, dk, dv = fat.attn_bwd(q, k, v, o, lse, do, causal, scale)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_forward_and_backward_replay_in_a_graph(cuda_device, d, causal):
    B, H, N, X = 2, 3, 700, 64
    scale = d ** -0.5
    q, k, v = (t.cuda() for t in gen.random_qkv(B, H, N, d, seed=901 + d))
    do = gen.random_qkv(B, H, N, d, seed=902 + d)[0].cuda()
    ref = _eager(q, k, v, do, causal, scale, X)

    # static buffers the graph reads and writes
    o = torch.empty_like(ref[0])
    lse = torch.empty_like(ref[1])
    grads = tuple(torch.empty_like(ref[2]) for _ in range(3))
    ws = torch.empty(fat.load_library().fat_attn_bwd_workspace_bytes(B, H, N),
                     dtype=torch.uint8, device=cuda_device)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capturing stream's kind of stream
        fat.attn_fwd(q, k, v, causal, scale, X, out=(o, lse))
        fat.attn_bwd(q, k, v, o, lse, do, causal, scale, workspace=ws, out=grads)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fat.attn_fwd(q, k, v, causal, scale, X, out=(o, lse))
        fat.attn_bwd(q, k, v, o, lse, do, causal, scale, workspace=ws, out=grads)

    for t in (o, lse, *grads):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert fat.check_device_error() == fat.FAT_OK
    got = (o, lse, *grads)
    for name, a, b in zip(("o", "lse", "dk", "dv"), (got[0], got[1], got[3], got[4]),
                          (ref[0], ref[1], ref[3], ref[4])):
        # the forward and dK, dV have a fixed order of operations
        assert torch.equal(a, b), name
    # dQ is summed by reduce-adds in no fixed order
    torch.testing.assert_close(got[2], ref[2], rtol=1e-5, atol=1e-5 * float(ref[2].abs().max()))

    # new inputs in the same buffers: the replay reads them
    q2, k2, v2 = (t.cuda() for t in gen.random_qkv(B, H, N, d, seed=903 + d))
    ref2 = _eager(q2, k2, v2, do, causal, scale, X)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref2[0]) and torch.equal(lse, ref2[1])
    assert torch.equal(grads[1], ref2[3]) and torch.equal(grads[2], ref2[4])
    torch.testing.assert_close(grads[0], ref2[2], rtol=1e-5,
                               atol=1e-5 * float(ref2[2].abs().max()))
