"""Test-side helpers: index permutations between the library's and the oracle's array orders,
layout views, and comparisons.  No method arithmetic lives here."""
import numpy as np
import torch

from block_scaled_causal_gb300 import inputs as I


def vsc_as_oracle(vsc: np.ndarray) -> np.ndarray:
    """The library's columnwise V scales [B,H,S/32,D] in the oracle's order [B,H,D,S/32]."""
    return np.ascontiguousarray(np.swapaxes(vsc, -1, -2))


def bshd_np(x: torch.Tensor, layout: int) -> np.ndarray:
    """CPU numpy copy of a tensor stored in `layout`, viewed as [B,S,H,D]."""
    t = I.to_bshd(x.cpu(), layout)
    if t.dtype == torch.bfloat16:
        t = t.float()
    return np.ascontiguousarray(t.numpy())


def as_f64(x: torch.Tensor) -> np.ndarray:
    return x.cpu().float().numpy().astype(np.float64)
