"""Workload shapes and seeded synthetic inputs.

This module is shared by the FP64 oracle side (tests, the CPU baseline) and the
CUDA side (tests, bench, smoke).  It holds no arithmetic of the attention method:
only the shapes of the workloads and the seeded random draws that both sides
consume.

Input recipe (the pages fix no seed or distribution, so this is a stated reading):
  * ``torch.Generator('cpu').manual_seed(seed)``;
  * draw q, k, v, dO in that order as float32 N(0, 1), natural token order,
    shape [B, H, T, D] (k and v use H_kv heads, q and dO use H_q heads);
  * optionally multiply q by ``q_scale`` after the draw (the stress case for
    safe softmax on the GPT-2-shaped workload);
  * cast to the workload dtype (bf16 rounding is torch's round-to-nearest-even).
The oracle consumes the cast values converted exactly to float64.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, dtype, context-parallel split."""

    name: str
    B: int
    H_q: int
    H_kv: int
    T: int
    D: int
    cp: int
    layout: str          # "contiguous" | "zigzag"
    dtype: str           # "f32" | "bf16"
    a2a: int = 1         # all-to-all group size (hierarchical a2a x p2p split)
    seed: int = 0
    q_scale: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def attended_pairs(self) -> int:
        """Causal (q, k) pairs with k <= q, over all batches and query heads."""
        return self.B * self.H_q * self.T * (self.T + 1) // 2

    @property
    def fwd_flops(self) -> float:
        # 2*d for q.k plus 2*d for p*v per attended pair
        return 4.0 * self.D * self.attended_pairs

    @property
    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny exactness case and shapes like the GPT-2 / LLaMA /
# Qwen3 attention layers plus a long-context sweep.
TINY = Workload("tiny_f32_T64", 1, 2, 2, 64, 16, 4, "contiguous", "f32")
GPT2 = Workload("gpt2_small_T1024", 4, 12, 12, 1024, 64, 2, "contiguous", "bf16")
LLAMA = Workload("llama_gqa_T8192_cp8_zigzag", 1, 32, 8, 8192, 128, 8, "zigzag", "bf16")
QWEN3 = Workload("qwen3_gqa_T32768_a2a2_p2p4_zigzag", 1, 32, 4, 32768, 128, 8, "zigzag",
                 "bf16", a2a=2)
LONG = Workload("long_T131072_zigzag", 1, 8, 8, 131072, 128, 8, "zigzag", "bf16")
# the full Ulysses mode (a2a = cp, so the ring has one rank): the LLaMA shape with the
# all-to-all over all 8 ranks, each then holding 4 query heads and 1 K/V head of the
# whole sequence
ULYSSES = Workload("llama_gqa_T8192_ulysses8", 1, 32, 8, 8192, 128, 8, "zigzag", "bf16", a2a=8)

GPT2_VARIANTS = [GPT2.replace(cp=cp, layout=lay, name=f"gpt2_small_T1024_cp{cp}_{lay}")
                 for cp in (2, 4) for lay in ("contiguous", "zigzag")]
GPT2_STRESS = GPT2.replace(seed=1, q_scale=4.0, name="gpt2_small_T1024_q4")
LONG_SWEEP = [LONG.replace(cp=cp, name=f"long_T131072_cp{cp}_zigzag") for cp in (4, 8, 16, 32)]

ALL = {w.name: w for w in [TINY, GPT2, LLAMA, QWEN3, LONG, ULYSSES, GPT2_STRESS,
                           *GPT2_VARIANTS, *LONG_SWEEP]}


def packed_starts(w: Workload, n_docs: int, seed: int = 1234) -> np.ndarray:
    """Seeded document starts int32 [B, n_docs + 1] for packed sequences: n_docs - 1
    distinct cut points drawn uniformly from 1..T-1, the same for every batch row."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, w.T), size=n_docs - 1, replace=False))
    row = np.concatenate([[0], cuts, [w.T]]).astype(np.int32)
    return np.tile(row, (w.B, 1))


def draw(w: Workload, seed: Optional[int] = None):
    """Seeded float32 draws (q, k, v, dO) in natural token order, [B, H, T, D]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    q = torch.randn((w.B, w.H_q, w.T, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.H_kv, w.T, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.H_kv, w.T, w.D), generator=g, dtype=torch.float32)
    do = torch.randn((w.B, w.H_q, w.T, w.D), generator=g, dtype=torch.float32)
    if w.q_scale != 1.0:
        q.mul_(w.q_scale)
    return q, k, v, do


def torch_dtype(w: Workload) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[w.dtype]


def draw_cast(w: Workload, seed: Optional[int] = None):
    """The draws cast to the workload dtype (what the GPU consumes)."""
    dt = torch_dtype(w)
    return tuple(x.to(dt) for x in draw(w, seed))


def as_f64(x: torch.Tensor):
    """Exact float64 copy as a numpy array (bf16 and f32 embed exactly)."""
    return x.detach().to("cpu").to(torch.float64).numpy()
