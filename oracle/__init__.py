"""CPU oracle for the fused attention forward pass (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and
``tensorized_online_softmax_gb300``) never imports it.

It wraps ``oracle.c`` (plain C, double precision, pthreads) through ctypes:

* :func:`attn_fwd`       -- the plain definition of softmax attention (the oracle);
* :func:`attn_fwd_qk`    -- the same for Nq query rows against Nk keys;
* :func:`attn_naive`     -- brute force in long double, full S materialised;
* :func:`attn_surrogate` -- Algorithm 1 of "FlashAttention-T: Towards Fully
  Tensorized Attention by Exploiting Tensor-Vector Parallelism" (section A2,
  tensorized online softmax) with the surrogate maximum over X-row tiles.

The backward pass's oracle (gradients of the same definition) is
:mod:`oracle.backward` (numpy, float64).

All arrays are float64 numpy arrays, row-major [B, H, N, d] (LSE [B, H, N]).
``scale`` is passed as a Python float; callers that mirror a float32 ABI
argument pass ``float(np.float32(scale))``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared"]


def build(force: bool = False, src: str = _SRC, out: str = _SO, extra_flags=()) -> str:
    """Compile ``oracle.c`` with gcc into ``oracle/_build/liboracle.so``."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.c_long


def load(path: str = _SO):
    """Load (building if needed) a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_available_cores.restype = ctypes.c_int
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [_D, _D, _D, _D, _D, _L, _L, _L, _L, ctypes.c_int,
                                    ctypes.c_double, _L, _L, _L, ctypes.c_int]
    lib.oracle_attn_fwd_qk.restype = ctypes.c_int
    lib.oracle_attn_fwd_qk.argtypes = [_D, _D, _D, _D, _D, _L, _L, _L, _L, _L, ctypes.c_int,
                                       ctypes.c_double, _L, _L, _L, ctypes.c_int]
    lib.oracle_attn_naive.restype = ctypes.c_int
    lib.oracle_attn_naive.argtypes = [_D, _D, _D, _D, _D, _L, _L, _L, _L, ctypes.c_int,
                                      ctypes.c_double]
    lib.oracle_attn_surrogate.restype = ctypes.c_long
    lib.oracle_attn_surrogate.argtypes = [_D, _D, _D, _D, _D, _D, _L, _L, _L, _L, ctypes.c_int,
                                          ctypes.c_double, _L, _L, _L]
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load()
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _as_f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor on the CPU
        a = a.detach().to("cpu").double().numpy()
    a = np.ascontiguousarray(a, dtype=np.float64)
    if a.ndim != 4:
        raise ValueError("expected a [B, H, N, d] array")
    return a


def available_cores() -> int:
    return int(_get().oracle_available_cores())


def attn_fwd(q, k, v, causal: bool, scale: float, rows: slice | None = None,
             nthreads: int = 0, lib=None):
    """Plain softmax attention in double precision.

    Returns ``(o, lse)``; with ``rows=slice(begin, end, step)`` only those query
    rows of every (b, h) are computed and the others are NaN.
    """
    lib = lib or _get()
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one shape")
    o = np.full((B, H, N, d), np.nan)
    lse = np.full((B, H, N), np.nan)
    if rows is None:
        rb, re_, rs = 0, N, 1
    else:
        rb, re_, rs = rows.indices(N)
    rc = lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                             int(bool(causal)), float(scale), rb, re_, rs, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    return o, lse


def attn_fwd_qk(q, k, v, causal: bool, scale: float, rows: slice | None = None,
                nthreads: int = 0, lib=None):
    """Plain softmax attention of Nq query rows against Nk keys, in double.

    q: [B, H, Nq, d]; k, v: [B, H, Nk, d].  Causal keeps key j for query i iff
    j <= i + Nk - Nq (the queries are the last Nq positions).
    """
    lib = lib or _get()
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] with q's B, H, d")
    o = np.full((B, H, Nq, d), np.nan)
    lse = np.full((B, H, Nq), np.nan)
    rb, re_, rs = (0, Nq, 1) if rows is None else rows.indices(Nq)
    rc = lib.oracle_attn_fwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                int(bool(causal)), float(scale), rb, re_, rs, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_qk failed ({rc})")
    return o, lse


def attn_naive(q, k, v, causal: bool, scale: float, lib=None):
    """Brute-force attention in long double (tiny inputs only)."""
    lib = lib or _get()
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    if N > 512:
        raise ValueError("the brute-force check is for tiny inputs")
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    rc = lib.oracle_attn_naive(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                               int(bool(causal)), float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_naive failed ({rc})")
    return o, lse


def attn_surrogate(q, k, v, causal: bool, scale: float, X: int, BM: int = 128, BN: int = 128,
                   lib=None):
    """Blocked online softmax with the X-row surrogate maximum, in double.

    Returns ``(o, lse, gap_log2, n_all_underflow)``; ``gap_log2`` holds, per row,
    log2(e) * (final surrogate maximum - exact row maximum).
    """
    lib = lib or _get()
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    gap = np.empty((B, H, N))
    n = lib.oracle_attn_surrogate(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(gap),
                                  B, H, N, d, int(bool(causal)), float(scale), X, BM, BN)
    if n < 0:
        raise RuntimeError(f"oracle_attn_surrogate failed ({n})")
    return o, lse, gap, int(n)
