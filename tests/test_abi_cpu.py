"""The C ABI library builds, loads, exports every entry point of
include/fat_attn.h, and rejects bad arguments before touching a GPU.
No compute call is made here (no GPU in this environment)."""
import ctypes
import os
import re
import subprocess

import pytest

import tensorized_online_softmax_gb300 as fat
from tensorized_online_softmax_gb300 import _build

HEADER = os.path.join(_build.ROOT, "include", "fat_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fat_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if _build.nvcc_path() is None and not os.path.exists(_build.LIB_PATH):
        pytest.skip("no nvcc and no prebuilt library")
    return fat.load_library()


def test_header_declares_the_abi():
    assert declared_functions() == sorted(fat.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True).stdout
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_no_symbol_is_unique_across_loaded_libraries(lib):
    # each loaded copy of the library must keep its own kernel launch state
    # (function-local statics of the kernel templates); GCC's STB_GNU_UNIQUE
    # binding would merge them across copies, so the build turns it off
    out = subprocess.run(["nm", "-D", _build.LIB_PATH], capture_output=True, text=True).stdout
    # (nm marks a unique global "u"; "U" is an undefined symbol)
    unique = [line for line in out.splitlines() if re.search(r"\su\s", line)]
    assert out.strip() and not unique, unique[:5]


def test_status_strings(lib):
    for code, name in [(0, "FAT_OK"), (-1, "FAT_ERR_INVALID_ARG"), (-2, "FAT_ERR_UNSUPPORTED"),
                       (-3, "FAT_ERR_ALIGNMENT"), (-4, "FAT_ERR_LAUNCH"),
                       (-5, "FAT_ERR_DEVICE_TIMEOUT"), (-6, "FAT_ERR_ARCH")]:
        assert lib.fat_status_string(code).decode() == name


def _fwd(lib, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, d=64,
         causal=0, scale=0.125, X=16, fn="fat_attn_fwd"):
    return getattr(lib, fn)(q, k, v, o, lse, B, H, N, d, causal, scale, X, None)


@pytest.mark.parametrize("fn", ["fat_attn_fwd", "fat_attn_fwd_vec"])
def test_validation_before_launch(lib, fn):
    assert _fwd(lib, q=None, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, lse=None, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, d=96, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, d=256, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, X=8, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, X=48, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, N=0, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, B=0, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, H=-1, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan"), fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, scale=-1.0, fn=fn) == fat.FAT_ERR_INVALID_ARG
    assert _fwd(lib, q=0x1001, fn=fn) == fat.FAT_ERR_ALIGNMENT
    assert _fwd(lib, o=0x4008, fn=fn) == fat.FAT_ERR_ALIGNMENT
    assert _fwd(lib, lse=0x5004, fn=fn) == fat.FAT_ERR_ALIGNMENT


def test_ex_validation(lib):
    assert lib.fat_attn_fwd_ex(None) == fat.FAT_ERR_INVALID_ARG
    p = fat.FatParams(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, d=64,
                      causal=0, scale=0.125, X=16, variant=7, dtype=0)
    assert lib.fat_attn_fwd_ex(ctypes.byref(p)) == fat.FAT_ERR_INVALID_ARG
    p.variant, p.dtype = 0, 9
    assert lib.fat_attn_fwd_ex(ctypes.byref(p)) == fat.FAT_ERR_INVALID_ARG


def test_z_mode_validation(lib):
    """Z on the tensor pipe exists for the tensorized variant, X = 128 and
    bf16 inputs only; other requests are refused before any device call."""
    base = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, d=128,
                causal=0, scale=0.125, X=128, variant=0, dtype=0)
    for kw, want in [(dict(z_mode=2), fat.FAT_ERR_INVALID_ARG),
                     (dict(z_mode=-1), fat.FAT_ERR_INVALID_ARG),
                     (dict(z_mode=1, X=64), fat.FAT_ERR_UNSUPPORTED),
                     (dict(z_mode=1, X=16), fat.FAT_ERR_UNSUPPORTED),
                     (dict(z_mode=1, variant=1), fat.FAT_ERR_UNSUPPORTED),
                     (dict(z_mode=1, dtype=2), fat.FAT_ERR_UNSUPPORTED),
                     (dict(z_mode=1, dtype=1, q_descale=1.0, k_descale=1.0, v_descale=1.0),
                      fat.FAT_ERR_UNSUPPORTED)]:
        p = fat.FatParams(**dict(base, **kw))
        assert lib.fat_attn_fwd_ex(ctypes.byref(p)) == want, kw


def test_block_mode_validation(lib):
    """Only the two block modes exist; anything else is refused before any
    device call."""
    base = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, d=128,
                causal=0, scale=0.125, X=128, variant=0, dtype=0)
    for bm in (2, -1, 99):
        p = fat.FatParams(**dict(base, block_mode=bm))
        assert lib.fat_attn_fwd_ex(ctypes.byref(p)) == fat.FAT_ERR_INVALID_ARG, bm
    assert fat.BLOCK_MODES == {"auto": 0, "per_tile": 1}


def test_params_struct_layout_matches_header(tmp_path):
    """ctypes mirror of fat_params has the C compiler's size and offsets."""
    cuda_inc = "/usr/local/cuda/include"
    if not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("CUDA headers not found")
    fields = [f[0] for f in fat.FatParams._fields_]
    src = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void){",
           'printf("%zu\\n", sizeof(fat_params));']
    src += [f'printf("%zu\\n", offsetof(fat_params, {f}));' for f in fields]
    src += ["return 0;}"]
    c = tmp_path / "layout.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", cuda_inc, "-o", str(exe), str(c)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(fat.FatParams)
    for f, off in zip(fields, vals[1:]):
        assert getattr(fat.FatParams, f).offset == off, f


def test_splitkv_workspace_and_validation(lib):
    ws = lib.fat_attn_splitkv_workspace_bytes
    # splits x B*H x Nq x (d + 1) fp32, plus alignment slack
    assert ws(2, 3, 5, 128, 4) == 4 * 6 * 5 * 129 * 4 + 256
    assert ws(1, 1, 1, 96, 2) == 0 and ws(1, 1, 1, 64, 0) == 0 and ws(1, 1, 1, 64, 65) == 0
    f = lib.fat_attn_fwd_splitkv
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, Nq=4, Nk=1024,
                d=128, causal=0, scale=0.1, X=128, splits=4, ws=None, wsb=0)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"],
                 a["d"], a["causal"], a["scale"], a["X"], a["splits"], a["ws"], a["wsb"], None)

    assert call() == fat.FAT_ERR_INVALID_ARG               # several ranges, no workspace
    assert call(ws=0x8000, wsb=16) == fat.FAT_ERR_INVALID_ARG  # workspace too small
    assert call(splits=0) == fat.FAT_ERR_INVALID_ARG
    assert call(splits=65) == fat.FAT_ERR_INVALID_ARG
    assert call(causal=1, Nq=2048, Nk=1024) == fat.FAT_ERR_INVALID_ARG  # Nk < Nq, causal
    assert call(Nk=0) == fat.FAT_ERR_INVALID_ARG


def test_bwd_validation(lib):
    """fat_attn_bwd refuses bad arguments before any device call."""
    ws_bytes = lib.fat_attn_bwd_workspace_bytes(2, 3, 300)
    # D and log2(e) LSE per row, rows padded to whole 128-row blocks
    assert ws_bytes == 2 * 2 * 3 * 384 * 4 + 256
    assert lib.fat_attn_bwd_workspace_bytes(0, 3, 300) == 0
    assert lib.fat_attn_bwd_workspace_bytes(1, 1, 0) == 0
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, do=0x6000, dq=0x7000,
                dk=0x8000, dv=0x9000, B=2, H=3, N=300, d=64, causal=1, scale=0.125, ws=0xA000,
                wsb=ws_bytes)

    def call(**kw):
        a = dict(args, **kw)
        return lib.fat_attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"],
                                a["dk"], a["dv"], a["B"], a["H"], a["N"], a["d"], a["causal"],
                                a["scale"], a["ws"], a["wsb"], None)

    for kw in (dict(q=None), dict(do=None), dict(dq=None), dict(ws=None), dict(d=96),
               dict(d=256), dict(N=0), dict(B=0), dict(H=-2), dict(scale=0.0),
               dict(scale=float("inf")), dict(wsb=ws_bytes - 1)):
        assert call(**kw) == fat.FAT_ERR_INVALID_ARG, kw
    for kw in (dict(q=0x1008), dict(do=0x6004), dict(dq=0x7004), dict(o=0x4008),
               dict(lse=0x5002)):
        assert call(**kw) == fat.FAT_ERR_ALIGNMENT, kw


def test_host_entry_validation(lib):
    """fat_attn_fwd_host refuses bad arguments before any device call."""
    ws = lib.fat_attn_fwd_host_workspace_bytes(2, 3, 300, 64, 2)
    # three slots of 2 heads: q, k, v bf16 + o fp32 + lse fp32, each 256-aligned
    rows = 2 * 300
    a = lambda x: (x + 255) // 256 * 256
    assert ws == 3 * (3 * a(rows * 64 * 2) + a(rows * 64 * 4) + a(rows * 4)) + 256
    assert lib.fat_attn_fwd_host_workspace_bytes(2, 3, 300, 96, 2) == 0
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=2, H=3, N=300, d=64,
                causal=0, scale=0.125, X=64, hc=2, ws=0x6000, wsb=ws)

    def call(**kw):
        c = dict(args, **kw)
        return lib.fat_attn_fwd_host(c["q"], c["k"], c["v"], c["o"], c["lse"], c["B"], c["H"],
                                     c["N"], c["d"], c["causal"], c["scale"], c["X"], c["hc"],
                                     c["ws"], c["wsb"], None)

    for kw in (dict(q=None), dict(o=None), dict(ws=None), dict(d=256), dict(N=0), dict(X=48),
               dict(scale=0.0), dict(wsb=ws - 1)):
        assert call(**kw) == fat.FAT_ERR_INVALID_ARG, kw
