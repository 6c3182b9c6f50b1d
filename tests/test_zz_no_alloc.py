"""The split-KV entry point that allocates nothing (its partial results live
in a fixed array inside the library) gives the same results as the regular
split-KV entry point with a caller-provided workspace.  It serves callers
that cannot allocate device memory when they call: a process whose device
memory all belongs to its own pool, or code that must not call cudaMalloc or
cudaFree because those can block or synchronise the device.

Called through the C ABI directly, twice in a row with different inputs (the
array is shared and keeps the previous call's contents), and once with a
request larger than the array, which must be refused.  This file is collected
last so that a run stopping at the first failure has run everything else."""
import ctypes

import pytest
import torch

import tensorized_online_softmax_gb300 as fat

from gpu_helpers import compare

pytestmark = pytest.mark.gpu


def _qkv(B, H, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16).cuda(),
            torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).cuda(),
            torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).cuda())


def _call_noalloc(lib, q, k, v, causal, scale, splits):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = torch.full((B, H, Nq, d), float("nan"), device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), device="cuda")
    st = lib.fat_attn_fwd_splitkv_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), B, H, Nq, Nk, d, int(causal), ctypes.c_float(scale),
        128, splits, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, o, lse


def test_noalloc_splitkv_matches_the_workspace_entry_point(cuda_device):
    lib = fat.load_library()
    scale = 128 ** -0.5
    shapes = [((2, 8, 4, 6000, 128), False, 12, 11), ((1, 4, 16, 4096, 128), True, 7, 12)]
    for (B, H, Nq, Nk, d), causal, splits, seed in shapes:  # two calls in a row
        q, k, v = _qkv(B, H, Nq, Nk, d, seed)
        need = lib.fat_attn_splitkv_workspace_bytes(B, H, Nq, d, splits)
        assert 0 < need <= (16 << 20)
        o_ref, lse_ref = fat.attn_fwd_splitkv(q, k, v, causal, scale, 128, splits)
        st, o, lse = _call_noalloc(lib, q, k, v, causal, scale, splits)
        assert st == fat.FAT_OK
        torch.cuda.synchronize()
        assert fat.check_device_error() == fat.FAT_OK
        compare(o.double().cpu().numpy(), lse.double().cpu().numpy(),
                o_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy(),
                what=f"no-alloc {B, H, Nq, Nk, d} causal={causal}")


def test_noalloc_refuses_requests_beyond_its_array(cuda_device):
    lib = fat.load_library()
    q, k, v = _qkv(1, 1, 1, 256, 128, seed=13)
    # 64 x 64 heads x 128 rows x 129 floats x 64 splits is far beyond 16 MiB
    B, H, Nq, Nk, d, splits = 64, 64, 128, 4096, 128, 64
    assert lib.fat_attn_splitkv_workspace_bytes(B, H, Nq, d, splits) > (16 << 20)
    st = lib.fat_attn_fwd_splitkv_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(q.data_ptr()), B, H, Nq, Nk, d, 0, ctypes.c_float(0.1), 128, splits,
        None)
    assert st == fat.FAT_ERR_INVALID_ARG
