"""Host-thread re-entrancy of the C ABI: the first call of every kernel
instance in a process sets up that instance's launch attributes once per
device.  Here eight host threads make the first calls of eight instances at
the same moment, each on a stream of its own, in a fresh child process (so
that no earlier test has set anything up).  Each result must equal the same
call repeated afterwards from one thread: bit for bit where the kernel's
arithmetic order is fixed (every forward instance; dK and dV), and within
the rounding of fp32 additions in no fixed order for dQ, which the backward
pass accumulates with reduce-adds."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import threading
import torch
import tensorized_online_softmax_gb300 as fat

torch.cuda.init()
lib = fat.load_library()  # loading launches nothing


def qkv(B, H, N, d, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn((B, H, N, d), generator=g).to(dtype).cuda() for _ in range(3))


q1, k1, v1 = qkv(1, 4, 1000, 128, 1)
q2, k2, v2 = qkv(2, 3, 777, 64, 2)
q3, k3, v3 = qkv(1, 2, 1300, 128, 3, torch.float16)
q4, k4, v4 = (t.to(torch.float8_e4m3fn) for t in qkv(1, 2, 900, 128, 4))
q5, k5, v5 = qkv(1, 2, 1100, 128, 5)
q6, k6, v6 = qkv(1, 2, 640, 64, 6)
# the backward pass's inputs, from instances (X = 64, 32) that none of the
# racing calls below uses
o5, l5 = fat.attn_fwd(q5, k5, v5, True, None, 64)
o6, l6 = fat.attn_fwd(q6, k6, v6, False, None, 32)
g = torch.Generator().manual_seed(7)
do5 = torch.randn(q5.shape, generator=g).to(torch.bfloat16).cuda()
do6 = torch.randn(q6.shape, generator=g).to(torch.bfloat16).cuda()
torch.cuda.synchronize()

ops = {
    "fwd bf16 d128 X128 causal": lambda s: fat.attn_fwd(q1, k1, v1, True, None, 128, stream=s),
    "fwd bf16 d64 X64": lambda s: fat.attn_fwd(q2, k2, v2, False, None, 64, stream=s),
    "fwd vec d128 X16": lambda s: fat.attn_fwd_vec(q1, k1, v1, False, None, 16, stream=s),
    "fwd fp16 d128 X32": lambda s: fat.attn_fwd(q3, k3, v3, True, None, 32, stream=s,
                                                dtype="fp16"),
    "fwd e4m3 d128 X128": lambda s: fat.attn_fwd(q4, k4, v4, False, None, 128, stream=s,
                                                 dtype="e4m3"),
    "splitkv d128": lambda s: fat.attn_fwd_splitkv(q1, k1, v1, False, None, 128, 3, stream=s),
    "bwd d128 causal": lambda s: fat.attn_bwd(q5, k5, v5, o5, l5, do5, True, stream=s),
    "bwd d64": lambda s: fat.attn_bwd(q6, k6, v6, o6, l6, do6, False, stream=s),
}
names = list(ops)
first, errors = {}, []
start = threading.Barrier(len(names))


def worker(name):
    try:
        s = torch.cuda.Stream()
        start.wait()
        with torch.cuda.stream(s):
            out = ops[name](s)
        s.synchronize()
        first[name] = out
    except Exception as e:  # reported below
        errors.append(f"{name}: {e!r}")


threads = [threading.Thread(target=worker, args=(n,)) for n in names]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
assert fat.check_device_error() == fat.FAT_OK

for name in names:
    again = ops[name](torch.cuda.current_stream())
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(first[name], again)):
        if name.startswith("bwd") and i == 0:  # dQ: reduce-adds in no fixed order
            tol = 1e-5 * float(b.abs().max()) + 1e-6
            err = float((a - b).abs().max())
            assert err <= tol, (name, "dq", err, tol)
        else:
            assert torch.equal(a, b), (name, i)
assert fat.check_device_error() == fat.FAT_OK
print("OK", len(names))
"""


def test_first_calls_from_eight_threads_at_once(cuda_device):
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "OK 8" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
