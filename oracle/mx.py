"""Test infrastructure only: plain CPU oracle for OCP-MX (MXFP8) block quantisation.

Nothing in the product path may import this module; only the tests, the smoke
check and the CPU-baseline leg of the benchmark use it.

What it follows
---------------
* "[PyTorch] Add causal MXFP8 attention without future-token leakage through V
  scales" (TransformerEngine PR #3865), Description: MXFP8 operands are E4M3
  element bytes with one shared power-of-two (E8M0) scale per 32 consecutive
  elements; Q and K share a scale along the head dimension (rowwise), V shares
  one along 32 consecutive tokens (columnwise), and the token-normalised V copy
  carries one power-of-two amplitude per token.
* "FROST SDPA fp8: block-scaled O epilogues" (cudnn-frontend PR #1088), Summary:
  "UE8M0 scale factor per 32 d" for the MXFP8 format.
* The pages do not restate the OCP Microscaling v1.0 conversion rule.  This
  module writes it out from the mathematics of that public specification:

    1. amax = max |x_k| over the k elements of a block (exact fp64 values of
       the bf16 inputs);
    2. e = floor(log2(amax)) - emax_elem, with emax_elem = 8 for E4M3
       (448 = 1.75 * 2**8); floor(log2) is read off frexp, exactly;
       e is clamped to [-127, 127]; amax == 0 gives e = -127;
    3. the scale byte is e + 127;
    4. each element is x_k * 2**-e (exact in fp64) rounded once to the E4M3
       grid, round-to-nearest-even, saturating to +-448 (never NaN), sign of
       zero kept;
    5. decode is e4m3_value * 2**e (exact).

  A block holding a NaN or an infinity gets scale byte 0xFF and element bytes
  0x7F (the E8M0 and E4M3 NaN codes).

  A second scale rule, "ceil", rounds the scale up instead so that no element saturates:
  e = ceil(log2(amax / 448)), the smallest e with amax * 2^-e <= 448.  The pages note that TE's
  own quantisation kernels, not the OCP text, chose its scales; covering the block maximum is the
  plain reading of that.  Everything else is unchanged.

Everything is fp64 numpy.  Element values are returned as float64 arrays;
bytes as uint8 arrays.
"""
from __future__ import annotations

import numpy as np

E4M3_EMAX = 8            # largest binade exponent of E4M3 ("fn" variant)
E4M3_MAX = 448.0         # 1.75 * 2**8
E4M3_MIN_NORMAL_EXP = -6  # 2**-6 is the smallest normal
E4M3_MANT_BITS = 3
E4M3_SUB_STEP = 2.0 ** -9  # subnormal spacing = 2**(min_normal_exp - mant_bits)
E8M0_BIAS = 127


def _floor_log2(a: np.ndarray) -> np.ndarray:
    """floor(log2(a)) for finite a > 0, exactly (frexp gives a = m * 2**ex, m in [0.5, 1))."""
    _, ex = np.frexp(a)
    return ex.astype(np.int64) - 1


def e4m3_round(y: np.ndarray) -> np.ndarray:
    """Round finite fp64 values onto the E4M3 grid: RNE, saturate to +-448, keep sign of zero."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    # Spacing of the grid at a: 2**(E - 3) for normals (E = floor(log2 a) >= -6), 2**-9 below.
    e = np.where(a >= 2.0 ** E4M3_MIN_NORMAL_EXP,
                 _floor_log2(np.where(a > 0, a, 1.0)), E4M3_MIN_NORMAL_EXP)
    step = np.ldexp(1.0, (e - E4M3_MANT_BITS).astype(np.int64))
    q = np.rint(a / step) * step          # a/step is exact; rint is round-half-to-even
    q = np.minimum(q, E4M3_MAX)           # satfinite
    return np.copysign(q, y)


def e4m3_encode(q: np.ndarray) -> np.ndarray:
    """Byte codes of values already on the E4M3 grid (finite, |q| <= 448); NaN -> 0x7F."""
    q = np.asarray(q, dtype=np.float64)
    nan = np.isnan(q)
    q = np.where(nan, 0.0, q)
    sign = np.signbit(q).astype(np.uint8) << 7
    a = np.abs(q)
    normal = a >= 2.0 ** E4M3_MIN_NORMAL_EXP
    E = _floor_log2(np.where(a > 0, a, 1.0))
    exp_field = np.where(normal, E + 7, 0)
    mant = np.where(normal,
                    np.ldexp(a, (-E).astype(np.int64)) * 8 - 8,   # (a / 2**E - 1) * 8
                    a / E4M3_SUB_STEP)
    mant_i = mant.astype(np.int64)
    if not np.all(mant_i == mant):
        raise ValueError("e4m3_encode: value not on the E4M3 grid")
    if np.any(exp_field > 15) or np.any((exp_field == 15) & (mant_i == 7)):
        raise ValueError("e4m3_encode: value beyond 448")
    code = sign | (exp_field.astype(np.uint8) << 3) | mant_i.astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """fp64 values of E4M3 ("fn": no infinities, S.1111.111 is NaN) byte codes."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    ef = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(ef == 0, m * E4M3_SUB_STEP, np.ldexp(1.0 + m / 8.0, ef - 7))
    val = np.where((ef == 15) & (m == 7), np.nan, val)
    return s * val


def e8m0_exponent(amax: np.ndarray, rule: str = "floor") -> np.ndarray:
    """Shared exponent e (scale = 2**e) for finite block maxima.

    rule "floor": the OCP MX rule for E4M3 elements, floor(log2 amax) - 8.
    rule "ceil": ceil(log2(amax / 448)): one more than "floor" exactly when amax exceeds
    448 * 2**("floor" exponent), i.e. when the significand of amax is above 1.75.
    """
    amax = np.asarray(amax, dtype=np.float64)
    fl = _floor_log2(np.where(amax > 0, amax, 1.0))
    e = fl - E4M3_EMAX
    if rule == "ceil":
        e = e + (np.where(amax > 0, amax, 1.0) > np.ldexp(E4M3_MAX / 256.0, fl)).astype(np.int64)
    elif rule != "floor":
        raise ValueError(rule)
    e = np.where(amax > 0, e, -E8M0_BIAS)
    return np.clip(e, -E8M0_BIAS, E8M0_BIAS)


def e8m0_decode(sb: np.ndarray) -> np.ndarray:
    """fp64 value 2**(byte - 127) of E8M0 scale bytes; 0xFF is NaN."""
    sb = np.asarray(sb, dtype=np.uint8).astype(np.int64)
    return np.where(sb == 0xFF, np.nan, np.ldexp(1.0, sb - E8M0_BIAS))


def mx_quantize(x: np.ndarray, k: int, rule: str = "floor") -> tuple[np.ndarray, np.ndarray]:
    """Quantise along the LAST axis in blocks of k consecutive elements (scale rule as in
    e8m0_exponent).

    Returns (element bytes with x's shape, scale bytes with shape x.shape[:-1] + (n/k,)).
    """
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    if n % k:
        raise ValueError("last axis must be a multiple of the block size")
    xb = x.reshape(x.shape[:-1] + (n // k, k))
    finite = np.all(np.isfinite(xb), axis=-1)
    amax = np.max(np.abs(np.where(np.isfinite(xb), xb, 0.0)), axis=-1)
    e = e8m0_exponent(amax, rule)
    y = np.ldexp(xb, -e[..., None])            # x * 2**-e, exact
    q = e4m3_round(np.where(np.isfinite(y), y, 0.0))
    codes = e4m3_encode(q)
    codes = np.where(finite[..., None], codes, np.uint8(0x7F)).astype(np.uint8)
    sbytes = np.where(finite, e + E8M0_BIAS, 0xFF).astype(np.uint8)
    return codes.reshape(x.shape), sbytes


def mx_dequantize(codes: np.ndarray, sbytes: np.ndarray, k: int) -> np.ndarray:
    """Inverse of mx_quantize along the last axis: e4m3(code) * 2**(scale - 127), exact in fp64."""
    v = e4m3_decode(codes)
    n = v.shape[-1]
    vb = v.reshape(v.shape[:-1] + (n // k, k))
    return (vb * e8m0_decode(sbytes)[..., None]).reshape(v.shape)


# ----------------------------------------------------------------------------------------------
# The three quantisations of the attention operands.  Arrays are in the canonical [B, S, H, D]
# order (a test turns SBHD data into this order before calling).

MX_BLOCK = 32


def quantize_rowwise(x: np.ndarray, rule: str = "floor"):
    """Q or K: one scale per 32 consecutive head-dim elements of each (b, s, h) row.

    Returns (bytes [B,S,H,D], scales [B,H,S,D/32]).
    """
    codes, sb = mx_quantize(x, MX_BLOCK, rule)           # sb: [B,S,H,D/32]
    return codes, np.ascontiguousarray(sb.transpose(0, 2, 1, 3))


def dequantize_rowwise(codes: np.ndarray, sc: np.ndarray) -> np.ndarray:
    return mx_dequantize(codes, np.ascontiguousarray(sc.transpose(0, 2, 1, 3)), MX_BLOCK)


def quantize_colwise(v: np.ndarray, rule: str = "floor"):
    """V columnwise: one scale per 32 consecutive tokens of each (b, h, d) column.

    Returns (bytes of V transposed to [B,H,D,S], scales [B,H,D,S/32]).
    """
    vt = np.ascontiguousarray(np.asarray(v, dtype=np.float64).transpose(0, 2, 3, 1))  # [B,H,D,S]
    return mx_quantize(vt, MX_BLOCK, rule)


def dequantize_colwise(codes_t: np.ndarray, sc: np.ndarray) -> np.ndarray:
    """Decoded V in [B,S,H,D] from transposed bytes [B,H,D,S] and scales [B,H,D,S/32]."""
    return np.ascontiguousarray(mx_dequantize(codes_t, sc, MX_BLOCK).transpose(0, 3, 1, 2))


def quantize_token_norm(v: np.ndarray, rule: str = "floor"):
    """Token-normalised V: one power-of-two amplitude per (b, s, h) token row of D elements.

    The pages fix only "one power-of-two amplitude per token"; the amplitude is chosen by the
    same MX rule with the block spanning the whole row (k = D).
    Returns (bytes [B,S,H,D], scales [B,H,S]).
    """
    v = np.asarray(v, dtype=np.float64)
    codes, sb = mx_quantize(v, v.shape[-1], rule)        # sb: [B,S,H,1]
    return codes, np.ascontiguousarray(sb[..., 0].transpose(0, 2, 1))


def dequantize_token_norm(codes: np.ndarray, sc: np.ndarray) -> np.ndarray:
    sb = np.ascontiguousarray(sc.transpose(0, 2, 1))[..., None]
    return mx_dequantize(codes, sb, codes.shape[-1])
