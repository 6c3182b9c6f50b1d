"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module only *draws* inputs; it holds none of the attention arithmetic.
Every tensor is produced on the CPU with a seeded ``torch.Generator`` in fp32,
then rounded (round-to-nearest-even) to the storage type, so that the CUDA
library and the CPU oracle see bit-identical values.

Workloads (names say what they are):

=========================  ==========================================================
``tiny``                   B1 H1 N128 d64, N(0,1), scale 1/8, non-causal, X=16
``b4h16n2048d128``         B4 H16 N2048 d128, N(0,1), scale 1/sqrt(128), X=64
``b4h16n2048d128_causal``  the same, causal
``b2h16n8192d128_causal``  B2 H16 N8192 d128, N(0,1), causal, X=128 (long sequence)
``stress_b1h32n16384d64``  B1 H32 N16384 d64, Q,K = 2.8 N(0,1) plus a +30-nat logit
                           shift for 1% of query rows on one random 128-key block
                           per head; V N(0,1); non-causal, X=64
``fp8_b4h16n4096d128``     B4 H16 N4096 d128, e4m3 from N(0,1) with per-tensor fp32
                           scales (amax / 448); non-causal, X=128
=========================  ==========================================================

The stress shift is written into the last coordinate of Q and K: Q[r, d-1] =
SHIFT_COORD for the chosen rows (0 elsewhere) and K[j, d-1] = SHIFT_COORD for
the chosen key block (0 elsewhere), so the kernel sees only Q, K and V.
With SHIFT_COORD = 15.5 (exact in bf16) the realised shift is
scale * 15.5**2 = 30.03 nats; 31.0 gives 120.1 nats (used to force the
all-underflow fallback).
"""
from __future__ import annotations

import dataclasses
import math

import torch

E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    X: int
    dtype: str = "bf16"  # "bf16", "fp16" or "e4m3"
    kind: str = "normal"  # "normal", "stress" or "growth"
    seed: int = 0
    shift_coord: float = 15.5  # stress only
    qk_std: float = 1.0
    growth_nats: float = 0.0  # growth only: logit added per 128-key tile

    @property
    def scale(self) -> float:
        # float32 value of 1/sqrt(d): the number the C ABI receives
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    @property
    def flops(self) -> float:
        """4 B H N^2 d, halved for causal (the extra row-sum MMA is not counted)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 64, False, 16, seed=1001),
    "b4h16n2048d128": Workload("b4h16n2048d128", 4, 16, 2048, 128, False, 64, seed=1002),
    "b4h16n2048d128_causal": Workload("b4h16n2048d128_causal", 4, 16, 2048, 128, True, 64,
                                      seed=1002),
    "b2h16n8192d128_causal": Workload("b2h16n8192d128_causal", 2, 16, 8192, 128, True, 128,
                                      seed=1003),
    "stress_b1h32n16384d64": Workload("stress_b1h32n16384d64", 1, 32, 16384, 64, False, 64,
                                      kind="stress", seed=1004, qk_std=2.8),
    "fp8_b4h16n4096d128": Workload("fp8_b4h16n4096d128", 4, 16, 4096, 128, False, 128,
                                   dtype="e4m3", seed=1005),
}


def _normal(shape, gen) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32)


def stress_choices(w: Workload, gen: torch.Generator):
    """Per head: one random 128-aligned key block and ceil(1% of N) query rows."""
    n_rows = math.ceil(0.01 * w.N)
    n_blocks = max(1, w.N // 128)
    blocks = torch.randint(0, n_blocks, (w.B, w.H), generator=gen)
    rows = torch.stack([torch.randperm(w.N, generator=gen)[:n_rows] for _ in range(w.B * w.H)])
    return blocks, rows.view(w.B, w.H, n_rows)


def make_inputs(w: Workload):
    """Return a dict with CPU tensors ``q, k, v`` in the storage dtype.

    bf16 workloads: ``q, k, v`` are torch.bfloat16.
    e4m3 workloads: ``q, k, v`` are torch.float8_e4m3fn and ``q_descale,
    k_descale, v_descale`` are the per-tensor fp32 scales (value = code * scale).
    Stress workloads also return ``shift_rows`` [B, H, R] and ``shift_block`` [B, H].
    """
    gen = torch.Generator().manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    q = _normal(shape, gen) * w.qk_std
    k = _normal(shape, gen) * w.qk_std
    v = _normal(shape, gen)
    out = {}
    if w.kind == "stress":
        blocks, rows = stress_choices(w, gen)
        q[..., w.d - 1] = 0.0
        k[..., w.d - 1] = 0.0
        for b in range(w.B):
            for h in range(w.H):
                q[b, h, rows[b, h], w.d - 1] = w.shift_coord
                j0 = int(blocks[b, h]) * 128
                k[b, h, j0:min(j0 + 128, w.N), w.d - 1] = w.shift_coord
        out["shift_rows"] = rows
        out["shift_block"] = blocks
    if w.kind == "growth":
        # every query gets coordinate d-1 = 1 and key j gets
        # growth_nats * (j // 128) / scale there, so each 128-key tile raises
        # the logits of all rows by growth_nats over the previous one
        q[..., w.d - 1] = 1.0
        tile = torch.arange(w.N, dtype=torch.float32) // 128
        k[..., w.d - 1] = (w.growth_nats / w.scale) * tile
    if w.dtype == "bf16":
        out.update(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v.to(torch.bfloat16))
    elif w.dtype == "fp16":
        out.update(q=q.to(torch.float16), k=k.to(torch.float16), v=v.to(torch.float16))
    elif w.dtype == "e4m3":
        for name, t in (("q", q), ("k", k), ("v", v)):
            s = float(t.abs().max()) / E4M3_MAX
            s = float(torch.tensor(s, dtype=torch.float32))
            code = (t / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
            out[name] = code
            out[name + "_descale"] = s
    else:
        raise ValueError(w.dtype)
    return out


def widened(inputs: dict, name: str) -> torch.Tensor:
    """Exact float64 value of an input tensor (e4m3 codes times their descale)."""
    t = inputs[name].to(torch.float64)
    if inputs[name].dtype == torch.float8_e4m3fn:
        t = t * inputs[name + "_descale"]
    return t


def random_qkv(B, H, N, d, seed, dtype=torch.bfloat16, std=1.0):
    """Plain N(0, std^2) inputs of an arbitrary shape (tests of edge cases)."""
    gen = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    return tuple((_normal(shape, gen) * std).to(dtype) for _ in range(3))
