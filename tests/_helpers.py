"""Test-side helpers: index permutations between the library's scale atoms and the oracle's compact
scale arrays, layout views, and comparisons.  No method arithmetic lives here."""
import numpy as np
import torch

from block_scaled_causal_gb300 import inputs as I


def row_atoms_to_compact(atoms: np.ndarray) -> np.ndarray:
    """[B,H,S/128,512] row atoms -> [B,H,S,4]; byte (s%32)*16 + ((s%128)//32)*4 + c."""
    B, H, T, _ = atoms.shape
    a = atoms.reshape(B, H, T, 32, 4, 4)              # (r, w, c), s%128 = 32 w + r
    return np.ascontiguousarray(a.transpose(0, 1, 2, 4, 3, 5)).reshape(B, H, T * 128, 4)


def col_atoms_to_compact(atoms: np.ndarray) -> np.ndarray:
    """[B,H,S/128,512] column atoms -> [B,H,D=128,S/32]; byte (d%32)*16 + (d//32)*4 + kb."""
    B, H, T, _ = atoms.shape
    a = atoms.reshape(B, H, T, 32, 4, 4)              # (r, w, kb), d = 32 w + r
    return np.ascontiguousarray(a.transpose(0, 1, 4, 3, 2, 5)).reshape(B, H, 128, T * 4)


def perm32():
    """Token order inside each 32-token block of the columnwise V bytes: byte x holds token
    8*((x%8)//2) + 2*(x//8) + x%2 (an involution)."""
    x = np.arange(32)
    return 8 * ((x % 8) // 2) + 2 * (x // 8) + x % 2


def vt_to_token_order(vt: np.ndarray) -> np.ndarray:
    """[.., S] columnwise V bytes in perm32 order -> token order."""
    S = vt.shape[-1]
    blocks = vt.reshape(vt.shape[:-1] + (S // 32, 32))
    return np.ascontiguousarray(blocks[..., perm32()]).reshape(vt.shape)


def bshd_np(x: torch.Tensor, layout: int) -> np.ndarray:
    """CPU numpy copy of a tensor stored in `layout`, viewed as [B,S,H,D]."""
    t = I.to_bshd(x.cpu(), layout)
    if t.dtype == torch.bfloat16:
        t = t.float()
    return np.ascontiguousarray(t.numpy())


def as_f64(x: torch.Tensor) -> np.ndarray:
    return x.cpu().float().numpy().astype(np.float64)
