"""Seeded synthetic inputs for blockwise causal attention under context parallelism.

This module holds the workload recipe only: shapes, seeds, random draws and the
rotary position embedding applied to Q/K before sharding.  It contains none of
the attention, merge or sharding arithmetic, and both the CUDA path's tests and
the fp64 oracle receive the very same arrays from it.

Recipe (the pages benchmark random bf16 tensors only, "On Context
Parallelism", Results and Conclusion; no dataset is involved):
  * q, k, v drawn i.i.d. N(0, 1) in float32 from torch.Generator('cpu')
    seeded with `seed`, in the order q, k, v, shapes [B,S,N,D] / [B,S,Nkv,D];
  * the S=32768 workload applies rotate-half RoPE (base 10000) to q and k by
    GLOBAL position, in float64 on the float32 draws;
  * values are then rounded once to bfloat16 (round to nearest even); the
    oracle reads those bf16 values exactly (as float32/float64).
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    N: int
    Nkv: int
    D: int
    C: int
    layout: str = "zigzag"  # or "contiguous"
    rope: bool = False
    fp32_inputs: bool = False  # the tiny case draws fp32 (rounded to bf16 for the tensor cores)
    relayout: bool = False     # also run the Ulysses relayout on this workload
    seed: int = 0

    @property
    def s(self) -> int:
        return self.S // self.C

    @property
    def t(self) -> int:
        return self.S // (2 * self.C)

    @property
    def causal_pairs(self) -> int:
        """Visible (query, key) pairs per (batch, head) for full causal attention."""
        return self.S * (self.S + 1) // 2

    @property
    def flops(self) -> float:
        """Algorithmic attention FLOPs: 4*D per visible pair (QK^T and PV, 2 per MAC)."""
        return 4.0 * self.B * self.N * self.D * self.causal_pairs


WORKLOADS = {
    "tiny": Workload("tiny", B=1, S=256, N=2, Nkv=2, D=64, C=2, fp32_inputs=True),
    "s4k": Workload("s4k", B=2, S=4096, N=16, Nkv=16, D=64, C=4, relayout=True),
    "s32k": Workload("s32k", B=1, S=32768, N=32, Nkv=32, D=128, C=4, rope=True),
    "s128k": Workload("s128k", B=1, S=131072, N=8, Nkv=8, D=128, C=8),
    # the >= 256K regime "On Context Parallelism" (Results and Conclusion)
    # reports on, with the S=131072 workload's heads and head size
    "s256k": Workload("s256k", B=1, S=262144, N=8, Nkv=8, D=128, C=8),
    "s256k_c16": Workload("s256k_c16", B=1, S=262144, N=8, Nkv=8, D=128, C=16),
}


def sweep_workloads():
    """B=1, N=16, D=128, S in {8192,16384,65536} x C in {2,4,8} x {contiguous, zigzag}."""
    out = []
    for S in (8192, 16384, 65536):
        for C in (2, 4, 8):
            for layout in ("contiguous", "zigzag"):
                out.append(Workload("sweep_S%d_C%d_%s" % (S, C, layout), B=1, S=S, N=16, Nkv=16,
                                    D=128, C=C, layout=layout))
    return out


def _rope_inplace_f64(x: np.ndarray, base: float = 10000.0, chunk: int = 2048) -> None:
    """Rotate-half rotary embedding by global position, in float64, in place.

    x: float64 [B, S, N, D]; dims (d, d + D/2) rotate by angle pos * base^(-2d/D).
    Input preparation only (the attention block applies RoPE before attention,
    "On Context Parallelism", Introduction); it is not part of the measured path.
    """
    B, S, N, D = x.shape
    half = D // 2
    inv = base ** (-(np.arange(half, dtype=np.float64) * 2.0) / D)
    for s0 in range(0, S, chunk):
        s1 = min(S, s0 + chunk)
        ang = np.arange(s0, s1, dtype=np.float64)[:, None] * inv[None, :]
        c = np.cos(ang)[None, :, None, :]
        s = np.sin(ang)[None, :, None, :]
        x1 = x[:, s0:s1, :, :half].copy()
        x2 = x[:, s0:s1, :, half:].copy()
        x[:, s0:s1, :, :half] = x1 * c - x2 * s
        x[:, s0:s1, :, half:] = x1 * s + x2 * c


def make_qkv(w: Workload):
    """Return (q, k, v) as torch bf16 CPU tensors [B,S,N,D] / [B,S,Nkv,D], and for
    the fp32-input workload also the unrounded fp32 draws (else None)."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = torch.randn(w.B, w.S, w.N, w.D, generator=g, dtype=torch.float32)
    k = torch.randn(w.B, w.S, w.Nkv, w.D, generator=g, dtype=torch.float32)
    v = torch.randn(w.B, w.S, w.Nkv, w.D, generator=g, dtype=torch.float32)
    if w.rope:
        for t in (q, k):
            a = t.numpy().astype(np.float64)
            _rope_inplace_f64(a)
            t.copy_(torch.from_numpy(a.astype(np.float32)))
    raw = (q.clone(), k.clone(), v.clone()) if w.fp32_inputs else None
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), raw


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 tensor to a float64 numpy array."""
    return t.float().numpy().astype(np.float64)


def sample_rows(w: Workload, n_random: int = 512, edge: int = 64, seed: int = 1) -> np.ndarray:
    """Deterministic query-row sample in GLOBAL positions: the first and last
    `edge` rows of every zigzag chunk plus `n_random` rows drawn with `seed`."""
    n_chunks = 2 * w.C
    t = w.S // n_chunks
    rows = []
    for c in range(n_chunks):
        e = min(edge, t)
        rows.extend(range(c * t, c * t + e))
        rows.extend(range((c + 1) * t - e, (c + 1) * t))
    rng = np.random.default_rng(seed)
    rows.extend(rng.integers(0, w.S, size=n_random).tolist())
    return np.unique(np.asarray(rows, dtype=np.int64))


def merge_inputs(B: int, Sq: int, N: int, D: int, seed: int = 2, neg_inf_frac: float = 0.0):
    """Stand-alone merge operands: o ~ N(0,1) fp32, lse ~ N(0,1) + log(Sq) fp32.

    With neg_inf_frac > 0 that fraction of the tile's rows get lse = -inf (rows
    a causal partial cannot see)."""
    g = torch.Generator("cpu").manual_seed(seed)
    o_acc = torch.randn(B, Sq, N, D, generator=g)
    o_t = torch.randn(B, Sq, N, D, generator=g)
    lse_acc = torch.randn(B, N, Sq, generator=g) + float(np.log(Sq))
    lse_t = torch.randn(B, N, Sq, generator=g) + float(np.log(Sq))
    if neg_inf_frac > 0:
        mask = torch.rand(B, N, Sq, generator=g) < neg_inf_frac
        lse_t[mask] = float("-inf")
    return o_acc, lse_acc, o_t, lse_t
