"""Two copies of the library in one process.

A process can end up with two copies of libfat_attn.so loaded side by side
(an application and a plug-in each shipping one, or an old and a rebuilt
copy).  Each copy sets up its own kernels on first use (the shared-memory
attribute of every kernel instance), so each must keep its own per-device
launch state: were that state shared, the second copy would skip the set-up
of its own kernels and fail to launch them.  In a fresh child process, the
same forward and backward calls through a second copy of the library must
succeed and give the first copy's results.
"""
import os
import shutil
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, sys
import torch
import tensorized_online_softmax_gb300 as fat

torch.cuda.init()
first = fat.load_library()
second = ctypes.CDLL(sys.argv[1])
P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
for lib in (first, second):
    lib.fat_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P]
    lib.fat_attn_fwd.restype = I
    lib.fat_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, ctypes.c_size_t, P]
    lib.fat_attn_bwd.restype = I
    lib.fat_attn_bwd_workspace_bytes.argtypes = [I, I, I]
    lib.fat_attn_bwd_workspace_bytes.restype = ctypes.c_size_t

g = torch.Generator().manual_seed(11)
B, H, N, d, X = 1, 3, 900, 128, 64
q, k, v, do = (torch.randn((B, H, N, d), generator=g).to(torch.bfloat16).cuda() for _ in range(4))
s = torch.cuda.current_stream().cuda_stream
out = {}
for name, lib in (("first", first), ("second", second)):
    o = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = lib.fat_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, N, d, 1, d ** -0.5, X, s)
    assert st == 0, (name, "forward", st)
    ws = torch.empty(lib.fat_attn_bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device="cuda")
    grads = [torch.empty_like(o) for _ in range(3)]
    st = lib.fat_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          do.data_ptr(), *(t.data_ptr() for t in grads), B, H, N, d, 1, d ** -0.5,
                          ws.data_ptr(), ws.numel(), s)
    assert st == 0, (name, "backward", st)
    torch.cuda.synchronize()
    out[name] = (o, lse, *grads)
a, b = out["first"], out["second"]
assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]), "forward differs"
assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4]), "dk / dv differ"
torch.testing.assert_close(a[2], b[2], rtol=1e-5, atol=1e-5 * float(a[2].abs().max()))
print("two copies ok")
"""


def test_a_second_copy_of_the_library_launches_its_own_kernels(tmp_path):
    import tensorized_online_softmax_gb300 as fat

    src = fat.load_library()._name
    copy = tmp_path / "libfat_attn_copy.so"
    shutil.copy(src, copy)
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", CHILD, str(copy)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "two copies ok" in r.stdout, r.stdout + r.stderr
