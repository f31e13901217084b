"""Seeded synthetic inputs for the attention forward (shared by tests, benchmark and smoke check).

This module draws numbers only; it holds none of the quantisation or attention arithmetic.

Recipe (the workloads of "[PyTorch] Add causal MXFP8 attention without future-token leakage
through V scales", Performance section: batch 1, 16 query heads, 4 or 16 KV heads, D = 128,
sequence lengths 8K-32K, BSHD or SBHD):

* Q, K, V (and dO) ~ N(0, 1), drawn in fp32 on the CPU with torch generators seeded 0, 1, 2
  (and 3), then rounded to bf16;
* "every7x16": V tokens s with (s + 1) % 7 == 0 are multiplied by 16 (all heads and d), so the
  shared V block scales differ inside a block;
* "heavy1pct": ceil(0.01 * S) token positions, the first entries of torch.randperm(S) under a
  generator seeded 1, have V multiplied by 64 (a heavy-tailed block amax).
"""
from __future__ import annotations

import dataclasses
import math

import torch

BSHD = 0
SBHD = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int = 128
    layout: int = BSHD
    v_pattern: str = "none"     # "none" | "every7x16" | "heavy1pct"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """Causal forward FLOPs, 2 * B * Hq * S^2 * D (the pages' convention)."""
        return 2.0 * self.B * self.Hq * self.S * self.S * self.D


WORKLOADS = {
    "tiny_s128_h2_every7x16": Workload("tiny_s128_h2_every7x16", 1, 128, 2, 2, v_pattern="every7x16"),
    "gqa_s8k_h16_kv4": Workload("gqa_s8k_h16_kv4", 1, 8192, 16, 4),
    "mha_s16k_h16_heavy1pct": Workload("mha_s16k_h16_heavy1pct", 1, 16384, 16, 16,
                                       v_pattern="heavy1pct"),
    "gqa_s32k_h16_kv4": Workload("gqa_s32k_h16_kv4", 1, 32768, 16, 4),
    "mha_b2_s32k_h16_sbhd": Workload("mha_b2_s32k_h16_sbhd", 2, 32768, 16, 16, layout=SBHD),
}


def _randn(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32)


def v_token_multipliers(S: int, pattern: str) -> torch.Tensor:
    """Per-token fp32 multiplier for V (1 everywhere except the pattern's tokens)."""
    mult = torch.ones(S, dtype=torch.float32)
    if pattern == "every7x16":
        s = torch.arange(S)
        mult[(s + 1) % 7 == 0] = 16.0
    elif pattern == "heavy1pct":
        g = torch.Generator().manual_seed(1)
        idx = torch.randperm(S, generator=g)[: math.ceil(0.01 * S)]
        mult[idx] = 64.0
    elif pattern != "none":
        raise ValueError(pattern)
    return mult


def to_layout(x_bshd: torch.Tensor, layout: int) -> torch.Tensor:
    """Contiguous copy of a [B,S,H,D] tensor in the requested memory layout."""
    if layout == BSHD:
        return x_bshd.contiguous()
    return x_bshd.permute(1, 0, 2, 3).contiguous()


def to_bshd(x: torch.Tensor, layout: int) -> torch.Tensor:
    """[B,S,H,D] view of a tensor stored in `layout`."""
    return x if layout == BSHD else x.permute(1, 0, 2, 3)


def make_qkv(w: Workload, seed_offset: int = 0, with_do: bool = False):
    """bf16 CPU tensors (q, k, v[, do]) in w.layout, plus their [B,S,H,D] views."""
    q = _randn((w.B, w.S, w.Hq, w.D), 0 + seed_offset)
    k = _randn((w.B, w.S, w.Hkv, w.D), 1 + seed_offset)
    v = _randn((w.B, w.S, w.Hkv, w.D), 2 + seed_offset)
    v = v * v_token_multipliers(w.S, w.v_pattern)[None, :, None, None]
    out = [to_layout(t.to(torch.bfloat16), w.layout) for t in (q, k, v)]
    if with_do:
        do = _randn((w.B, w.S, w.Hq, w.D), 3 + seed_offset)
        out.append(to_layout(do.to(torch.bfloat16), w.layout))
    return tuple(out)
