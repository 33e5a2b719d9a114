"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no attention arithmetic: it only draws random numbers and
rounds them to bf16, so the oracle and the GPU path read the same bytes.

Recipe (one call = one problem):
  * generator: ``numpy.random.default_rng(seed)`` (PCG64);
  * draw order: Q ``[B,H,Nq,D]``, K ``[B,H,Nk,D]``, V ``[B,H,Nk,D]``,
    dO ``[B,H,Nq,D]``, each ``standard_normal`` in float32;
  * multiply every tensor by ``factor`` and Q, K additionally by
    ``qk_factor`` (the "x8" stability variant);
  * round to bf16 round-to-nearest-even (torch's ``.to(torch.bfloat16)``).

The shapes and distributions mirror the sweeps of the pages: i.i.d. N(0,1)
Q/K/V with B=8, H=1 and D in {16..128}, N in {256..16384}
("FlashAttention-2实现与优化：高效注意力机制详解", §2.1 benchmark sweep), and the
multi-head / long-context layer shapes used for measurement.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Problem:
    B: int
    H: int
    Nq: int
    Nk: int
    D: int
    causal: bool
    factor: float = 1.0
    qk_factor: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def name(self) -> str:
        s = f"B{self.B}H{self.H}q{self.Nq}k{self.Nk}D{self.D}{'c' if self.causal else 'n'}"
        if self.factor != 1.0:
            s += f"f{self.factor:g}"
        if self.qk_factor != 1.0:
            s += f"x{self.qk_factor:g}"
        return s


def draw(p: Problem, seed: int):
    """Return (q, k, v, do) as CPU bf16 torch tensors, contiguous [B,H,N,D]."""
    rng = np.random.default_rng(seed)
    shapes = [(p.B, p.H, p.Nq, p.D), (p.B, p.H, p.Nk, p.D),
              (p.B, p.H, p.Nk, p.D), (p.B, p.H, p.Nq, p.D)]
    out = []
    for i, shp in enumerate(shapes):
        x = rng.standard_normal(shp, dtype=np.float32)
        f = p.factor * (p.qk_factor if i < 2 else 1.0)
        if f != 1.0:
            x *= np.float32(f)
        out.append(torch.from_numpy(x).to(torch.bfloat16).contiguous())
    return tuple(out)


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact upcast of a bf16 tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()


# The five workloads (and the sweep) that parity covers; the fourth is the
# multi-head LLM-shaped layer that the benchmark times.
SMALL = Problem(B=8, H=1, Nq=256, Nk=256, D=16, causal=False)
SWEEP = [Problem(B=8, H=1, Nq=n, Nk=n, D=d, causal=c)
         for d in (16, 32, 64, 128) for n in (256, 1024, 4096) for c in (False, True)]
SWEEP_X8 = [dataclasses.replace(p, qk_factor=8.0) for p in SWEEP]
LONG = [Problem(B=8, H=1, Nq=n, Nk=n, D=d, causal=True) for n in (8192, 16384) for d in (64, 128)]
LAYER = Problem(B=4, H=32, Nq=4096, Nk=4096, D=128, causal=True, factor=0.5)
LONG_RAGGED = Problem(B=1, H=8, Nq=65537, Nk=65537, D=128, causal=True)


def flops_fwd(p: Problem) -> float:
    """Forward FLOPs by the 4*B*H*Nq*Nk*D convention, halved when causal."""
    f = 4.0 * p.B * p.H * p.Nq * p.Nk * p.D
    return f / 2 if p.causal else f


def flops_bwd(p: Problem) -> float:
    """Backward FLOPs: 2.5x the forward convention."""
    return 2.5 * flops_fwd(p)


def draw_varlen(lens_q, lens_k, H: int, D: int, seed: int, factor: float = 1.0):
    """Packed variable-length batch: Q, K, V, dO as bf16 [total, H, D] drawn like `draw`
    (standard normal float32, order Q, K, V, dO, times `factor`, bf16 RN) plus the
    int32 offsets cu_q, cu_k (B + 1 entries, starting at 0)."""
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    rng = np.random.default_rng(seed)
    out = []
    for n in (int(cu_q[-1]), int(cu_k[-1]), int(cu_k[-1]), int(cu_q[-1])):
        x = rng.standard_normal((n, H, D), dtype=np.float32)
        if factor != 1.0:
            x *= np.float32(factor)
        out.append(torch.from_numpy(x).to(torch.bfloat16).contiguous())
    return (*out, torch.from_numpy(cu_q), torch.from_numpy(cu_k))


def doc_lengths(total: int, seed: int, median: float = 1024.0, lo: int = 16, hi: int = 8192) -> list[int]:
    """Sequence lengths of a packed batch of documents: log-normal (sigma 1) around
    `median`, clipped to [lo, hi], drawn until they fill `total` tokens (the last one
    cut to fit)."""
    rng = np.random.default_rng(seed)
    lens, left = [], total
    while left > 0:
        n = int(np.clip(np.exp(rng.normal(np.log(median), 1.0)), lo, hi))
        n = min(n, left)
        lens.append(n)
        left -= n
    return lens


def flops_varlen(lens_q, lens_k, H: int, D: int, causal: bool, backward: bool = False) -> float:
    """FLOPs of a packed batch: the dense convention summed over its sequences."""
    f = sum(4.0 * H * nq * nk * D * (0.5 if causal else 1.0) for nq, nk in zip(lens_q, lens_k))
    return 2.5 * f if backward else f


# Packed batch of documents, 16384 tokens (the token count of the 4 x 4096 layer) with
# 32 heads of D = 128, causal within each document.
VARLEN_DOCS = dict(lens=doc_lengths(16384, seed=7), H=32, D=128, causal=True, factor=0.5)

