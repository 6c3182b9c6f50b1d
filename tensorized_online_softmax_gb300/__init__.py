"""GB300 (sm_103a) fused attention forward with the tensorized online softmax.

Thin Python binding over the C ABI of ``include/fat_attn.h`` (ctypes).  Every
step of the computation runs in the CUDA library; this module only checks
tensor shapes/dtypes, allocates the outputs with torch and marshals the
arguments.  There is no CPU fallback: if the CUDA library cannot be loaded,
every call raises.

The operation is the fused attention flow of "FlashAttention-T: Towards Fully
Tensorized Attention by Exploiting Tensor-Vector Parallelism" (papercache.org
summary, section A3 / Fig. 2) with its tensorized online softmax (section A2,
Algorithm 1); ``variant="vec"`` is the vector-softmax ablation arm.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "FatError", "load_library", "attn_fwd", "attn_fwd_vec", "attn_fwd_fp8", "attn_fwd_splitkv",
    "attn_bwd", "attn_fwd_host",
    "check_device_error", "status_string", "ABI_SYMBOLS", "FAT_OK",
    "FAT_ERR_INVALID_ARG", "FAT_ERR_UNSUPPORTED", "FAT_ERR_ALIGNMENT", "FAT_ERR_LAUNCH",
    "FAT_ERR_DEVICE_TIMEOUT", "FAT_ERR_ARCH",
]

FAT_OK = 0
FAT_ERR_INVALID_ARG = -1
FAT_ERR_UNSUPPORTED = -2
FAT_ERR_ALIGNMENT = -3
FAT_ERR_LAUNCH = -4
FAT_ERR_DEVICE_TIMEOUT = -5
FAT_ERR_ARCH = -6

VARIANTS = {"tensor": 0, "vec": 1}
DTYPES = {"bf16": 0, "e4m3": 1, "fp16": 2}
LMODES = {"vector": 0, "tensor": 1}
BLOCK_MODES = {"auto": 0, "per_tile": 1}
ZMODES = {"vector": 0, "tensor": 1}
TRACE_ITERS = 128
TRACE_EVENTS = 5
TRACE_WORDS = TRACE_EVENTS * 2 * TRACE_ITERS + 2

# every extern "C" entry point declared in include/fat_attn.h
ABI_SYMBOLS = (
    "fat_attn_fwd", "fat_attn_fwd_vec", "fat_attn_fwd_fp8", "fat_attn_fwd_splitkv",
    "fat_attn_splitkv_workspace_bytes", "fat_attn_splitkv_default_splits",
    "fat_attn_fwd_splitkv_noalloc", "fat_attn_fwd_ex",
    "fat_attn_bwd", "fat_attn_bwd_workspace_bytes",
    "fat_attn_fwd_host", "fat_attn_fwd_host_workspace_bytes",
    "fat_status_string", "fat_check_device_error",
)


class FatError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else
                         f"{status_string(status)} ({status})")


class FatParams(ctypes.Structure):
    """Mirror of ``fat_params`` in include/fat_attn.h (same field order)."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("d", ctypes.c_int),
        ("causal", ctypes.c_int), ("scale", ctypes.c_float), ("X", ctypes.c_int),
        ("variant", ctypes.c_int), ("dtype", ctypes.c_int), ("l_mode", ctypes.c_int),
        ("q_descale", ctypes.c_float), ("k_descale", ctypes.c_float),
        ("v_descale", ctypes.c_float),
        ("underflow_log2_threshold", ctypes.c_float),
        ("fallback_rows", ctypes.c_void_p),
        ("wait_poll_limit", ctypes.c_ulonglong),
        ("wait_timeout_ns", ctypes.c_ulonglong),
        ("stream", ctypes.c_void_p),
        ("trace", ctypes.c_void_p),
        ("z_mode", ctypes.c_int),
        ("block_mode", ctypes.c_int),
    ]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = True):
    """Load the in-tree CUDA library (building it first if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if build_if_missing and _build.is_stale(path) and _build.nvcc_path() is not None:
            _build.build()
        if not os.path.exists(path):
            raise FatError(FAT_ERR_LAUNCH, f"CUDA library {path} is missing; run build()")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I, F = ctypes.c_int, ctypes.c_float
        fwd_args = [P, P, P, P, P, I, I, I, I, I, F, I, P]
        for name in ("fat_attn_fwd", "fat_attn_fwd_vec"):
            getattr(lib, name).argtypes = fwd_args
            getattr(lib, name).restype = I
        lib.fat_attn_fwd_fp8.argtypes = [P, P, P, F, F, F, P, P, I, I, I, I, I, F, I, P]
        lib.fat_attn_fwd_fp8.restype = I
        lib.fat_attn_fwd_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, P,
                                             ctypes.c_size_t, P]
        lib.fat_attn_fwd_splitkv.restype = I
        lib.fat_attn_splitkv_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.fat_attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.fat_attn_splitkv_default_splits.argtypes = [I, I, I, I]
        lib.fat_attn_splitkv_default_splits.restype = I
        lib.fat_attn_fwd_splitkv_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, P]
        lib.fat_attn_fwd_splitkv_noalloc.restype = I
        lib.fat_attn_fwd_ex.argtypes = [ctypes.POINTER(FatParams)]
        lib.fat_attn_fwd_ex.restype = I
        lib.fat_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P,
                                     ctypes.c_size_t, P]
        lib.fat_attn_bwd.restype = I
        lib.fat_attn_bwd_workspace_bytes.argtypes = [I, I, I]
        lib.fat_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fat_attn_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P,
                                          ctypes.c_size_t, P]
        lib.fat_attn_fwd_host.restype = I
        lib.fat_attn_fwd_host_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.fat_attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.fat_status_string.argtypes = [I]
        lib.fat_status_string.restype = ctypes.c_char_p
        lib.fat_check_device_error.argtypes = [P]
        lib.fat_check_device_error.restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    names = {0: "FAT_OK", -1: "FAT_ERR_INVALID_ARG", -2: "FAT_ERR_UNSUPPORTED",
             -3: "FAT_ERR_ALIGNMENT", -4: "FAT_ERR_LAUNCH", -5: "FAT_ERR_DEVICE_TIMEOUT",
             -6: "FAT_ERR_ARCH"}
    return names.get(status, "FAT_ERR_UNKNOWN")


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_inputs(q, k, v, dtypes):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype not in dtypes:
            raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k and v must have the same shape")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k and v must be on one device")


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, X: int = 64,
             variant: str = "tensor", *, out=None, stream=None, fallback_rows=None,
             underflow_log2_threshold: float = 0.0, wait_poll_limit: int = 0,
             wait_timeout_ns: int = 0, dtype: str = "bf16", descales=(1.0, 1.0, 1.0),
             l_mode: str = "vector", trace=None, z_mode: str = "vector",
             block_mode: str = "auto"):
    """Fused attention forward.  Returns ``(o, lse)`` (fp32 [B,H,N,d], fp32 [B,H,N]).

    ``q, k, v``: contiguous CUDA tensors [B, H, N, d] (bf16; fp16 with
    ``dtype="fp16"``; or float8_e4m3fn with ``dtype="e4m3"`` and per-tensor
    ``descales``).  ``scale`` defaults to
    1/sqrt(d).  ``fallback_rows`` is an optional int32 CUDA tensor of one
    element that the kernel increments by the number of rows it recomputed.
    ``l_mode="tensor"`` forms the row sum on the tensor pipe (see fat_lmode in
    include/fat_attn.h for its accuracy); ``z_mode="tensor"`` has the S MMA
    subtract a reference offset (fat_zmode: bf16, X = 128, tensorized only).
    ``block_mode="per_tile"`` launches one thread block per 128-row query tile
    instead of one per SM taking tiles in turn (fat_block_mode).
    The call is asynchronous on ``stream`` (default: torch's current stream).
    """
    import torch

    lib = load_library()
    allowed = {"bf16": (torch.bfloat16,), "fp16": (torch.float16,),
               "e4m3": (torch.float8_e4m3fn,)}[dtype]
    _check_inputs(q, k, v, allowed)
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        o = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    p = FatParams()
    p.q, p.k, p.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    p.o, p.lse = o.data_ptr(), lse.data_ptr()
    p.B, p.H, p.N, p.d = B, H, N, d
    p.causal = int(bool(causal))
    p.scale = float(scale)
    p.X = int(X)
    p.variant = VARIANTS[variant]
    p.dtype = DTYPES[dtype]
    p.l_mode = LMODES[l_mode]
    p.z_mode = ZMODES[z_mode]
    p.block_mode = BLOCK_MODES[block_mode]
    p.q_descale, p.k_descale, p.v_descale = (float(x) for x in descales)
    p.underflow_log2_threshold = float(underflow_log2_threshold)
    p.fallback_rows = fallback_rows.data_ptr() if fallback_rows is not None else None
    p.wait_poll_limit = int(wait_poll_limit)
    p.wait_timeout_ns = int(wait_timeout_ns)
    p.stream = _stream_handle(stream).value
    p.trace = trace.data_ptr() if trace is not None else None
    with torch.cuda.device(q.device):
        st = lib.fat_attn_fwd_ex(ctypes.byref(p))
    if st != FAT_OK:
        raise FatError(st, "fat_attn_fwd_ex")
    return o, lse


def attn_fwd_vec(q, k, v, causal: bool = False, scale: float | None = None, X: int = 64, **kw):
    """Vector-softmax ablation variant (exact per-row maximum, vector row sum)."""
    return attn_fwd(q, k, v, causal, scale, X, variant="vec", **kw)


def attn_fwd_fp8(q, k, v, q_descale: float, k_descale: float, v_descale: float,
                 causal: bool = False, scale: float | None = None, X: int = 128, **kw):
    """e4m3 inputs with per-tensor descales; fp32 accumulation and outputs."""
    return attn_fwd(q, k, v, causal, scale, X, dtype="e4m3",
                    descales=(q_descale, k_descale, v_descale), **kw)


def attn_fwd_splitkv(q, k, v, causal: bool = False, scale: float | None = None, X: int = 128,
                     num_splits: int | None = None, *, workspace=None, out=None, stream=None):
    """Split-KV forward: q [B, H, Nq, d] against k, v [B, H, Nk, d] (bf16).

    The key range is split across thread blocks and the partial results are
    merged by LSE weights.  ``num_splits=None`` picks about one block per SM.
    ``workspace`` (a CUDA uint8 tensor) is allocated here if not given.
    Returns ``(o, lse)``.
    """
    import torch

    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a bf16 CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D tensor")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] with q's B, H, d")
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(q.device):
        if num_splits is None:
            num_splits = lib.fat_attn_splitkv_default_splits(B, H, Nq, Nk)
        nbytes = lib.fat_attn_splitkv_workspace_bytes(B, H, Nq, d, int(num_splits))
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        if out is None:
            o = torch.empty((B, H, Nq, d), dtype=torch.float32, device=q.device)
            lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
        else:
            o, lse = out
        st = lib.fat_attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, Nq, Nk, d, int(bool(causal)),
                                      float(scale), int(X), int(num_splits),
                                      workspace.data_ptr(), workspace.numel(),
                                      _stream_handle(stream))
    if st != FAT_OK:
        raise FatError(st, "fat_attn_fwd_splitkv")
    return o, lse


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, *,
             workspace=None, out=None, stream=None):
    """Backward pass: gradients of sum(O * dout) with respect to q, k, v.

    ``q, k, v, dout``: contiguous bf16 CUDA tensors [B, H, N, d]; ``o, lse``:
    the fp32 outputs of a forward call on the same inputs.  ``workspace`` (a
    CUDA uint8 tensor) is allocated here if not given.  Returns fp32
    ``(dq, dk, dv)``.
    """
    import torch

    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a bf16 CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    B, H, N, d = q.shape
    if (o.dtype != torch.float32 or o.shape != q.shape or not o.is_contiguous() or
            lse.dtype != torch.float32 or lse.shape != (B, H, N) or not lse.is_contiguous()):
        raise ValueError("o must be fp32 [B, H, N, d] and lse fp32 [B, H, N]")
    if scale is None:
        scale = d ** -0.5
    with torch.cuda.device(q.device):
        nbytes = lib.fat_attn_bwd_workspace_bytes(B, H, N)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        if out is None:
            dq, dk, dv = (torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
                          for _ in range(3))
        else:
            dq, dk, dv = out
        st = lib.fat_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                              workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if st != FAT_OK:
        raise FatError(st, "fat_attn_bwd")
    return dq, dk, dv


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, X: int = 64, *,
                  out=None, workspace=None, heads_per_chunk: int = 0, stream=None, device=None):
    """Forward pass on host-resident tensors (``fat_attn_fwd_host``).

    ``q, k, v``: contiguous bf16 CPU tensors [B, H, N, d] in page-locked memory
    (``tensor.pin_memory()``); ``out``: optional page-locked fp32 ``(o, lse)``.
    The problem is streamed through the device in chunks of heads, the copies
    overlapping the kernels.  ``workspace`` (a CUDA uint8 tensor) is
    allocated here if not given.  The call is asynchronous on ``stream``;
    synchronise it before reading ``o`` and ``lse``.  Returns ``(o, lse)``.
    """
    import torch

    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if (not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16 or
                not t.is_pinned()):
            raise ValueError(f"{name} must be a page-locked bf16 host tensor")
        if t.dim() != 4 or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if out is None:
        o = torch.empty((B, H, N, d), dtype=torch.float32).pin_memory()
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    else:
        o, lse = out
    for name, t, shape in (("o", o, (B, H, N, d)), ("lse", lse, (B, H, N))):
        if t.is_cuda or t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_pinned():
            raise ValueError(f"{name} must be a page-locked fp32 host tensor of shape {shape}")
    with torch.cuda.device(dev):
        nbytes = lib.fat_attn_fwd_host_workspace_bytes(B, H, N, d, int(heads_per_chunk))
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        st = lib.fat_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                   int(X), int(heads_per_chunk), workspace.data_ptr(),
                                   workspace.numel(), _stream_handle(stream))
    if st != FAT_OK:
        raise FatError(st, "fat_attn_fwd_host")
    return o, lse


def check_device_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error status."""
    lib = load_library()
    return lib.fat_check_device_error(_stream_handle(stream))


def raw_call(name: str, *args):
    """Call a C entry point by name with raw arguments (ABI tests)."""
    lib = load_library()
    return getattr(lib, name)(*args)
