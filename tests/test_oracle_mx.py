"""Pins for the oracle's MXFP8 quantiser (CPU only).

Each test checks the oracle against something other than itself: hand-computed blocks, an
independent table-search encoder built on torch's float8_e4m3fn decoding, torch's own fp32 ->
float8_e4m3fn cast for in-range values, and closed forms of the scale rule.
"""
import os

import numpy as np
import pytest
import torch

from oracle import mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_worked_examples.txt")


def _bf16_from_bits(bits):
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).view(np.int16)).view(torch.bfloat16)
    return t.float().numpy().astype(np.float64)


def _load_golden():
    blocks = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        parts = line.split()
        blk = blocks.setdefault(parts[0], {"in": [], "scale": None})
        if parts[1] == "in":
            blk["in"].append((int(parts[2], 16), int(parts[3], 16)))
        else:
            blk["scale"] = int(parts[2], 16)
    return blocks


@pytest.mark.parametrize("name", list(_load_golden().keys()))
def test_worked_examples(name):
    blk = _load_golden()[name]
    bits = np.zeros(32, dtype=np.uint16)
    want = np.zeros(32, dtype=np.uint8)
    for idx, (b, e) in enumerate(blk["in"]):
        bits[idx] = b
        want[idx] = e
    x = _bf16_from_bits(bits)
    codes, sb = mx.mx_quantize(x[None, :], 32)
    assert sb[0, 0] == blk["scale"], (name, hex(sb[0, 0]))
    np.testing.assert_array_equal(codes[0], want)


def _torch_e4m3_table():
    """Values of all 256 E4M3 byte codes as decoded by torch (independent of the oracle)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_table():
    codes = np.arange(256, dtype=np.uint8)
    ours = mx.e4m3_decode(codes)
    ref = _torch_e4m3_table()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    # sign of zero
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def _table_encode(y):
    """Independent encoder: nearest finite E4M3 code by exhaustive search, ties to even
    mantissa, saturating at +-448, sign of zero kept."""
    table = _torch_e4m3_table()
    finite_codes = np.array([c for c in range(256) if not np.isnan(table[c])])
    vals = table[finite_codes]
    out = np.empty(len(y), dtype=np.uint8)
    for n, v in enumerate(y):
        a = min(abs(v), 448.0)
        pos = finite_codes[(vals >= 0) & ~np.signbit(vals)]
        pv = table[pos]
        d = np.abs(pv - a)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if (pos[b] & 1) == 0]
        code = int(pos[best[0]])
        if np.signbit(v):
            code |= 0x80
        out[n] = code
    return out


def test_exhaustive_bf16_against_table_encoder():
    # every finite bf16 value, scaled into the E4M3 range by a few fixed exponents
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = _bf16_from_bits(bits)
    x = x[np.isfinite(x)]
    rng = np.random.default_rng(0)
    for e in (-7, 0, 5, -120, 100):
        y = np.ldexp(x, -e)
        # restrict to the range where the scale could have been chosen by the MX rule
        sel = np.abs(y) < 1024.0
        ys = y[sel]
        pick = rng.choice(len(ys), size=min(len(ys), 6000), replace=False)
        ys = ys[pick]
        ours = mx.e4m3_encode(mx.e4m3_round(ys))
        np.testing.assert_array_equal(ours, _table_encode(ys))


def test_in_range_matches_torch_cast():
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest even; beyond 448 it does not
    # saturate, so compare on |y| <= 448 only.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = _bf16_from_bits(bits)
    x = x[np.isfinite(x)]
    for e in (-8, -3, 0, 4):
        y = np.ldexp(x, -e)
        y = y[np.abs(y) <= 448.0]
        ref = torch.tensor(y, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        ours = mx.e4m3_encode(mx.e4m3_round(y))
        np.testing.assert_array_equal(ours, ref)


@pytest.mark.parametrize("k", [0, 1, 7, -5, -60, 100])
def test_scale_rule_binade_closed_form(k):
    # amax in [2^(k+8), 2^(k+9)) gives scale byte 127 + k; the bottom and top of the binade
    lo = np.ldexp(1.0, k + 8)
    hi = np.ldexp(1.0, k + 9) * (1 - 2.0 ** -8)       # largest bf16 below 2^(k+9)
    for amax in (lo, hi, np.ldexp(1.5, k + 8)):
        x = np.zeros((1, 32))
        x[0, 3] = -amax
        _, sb = mx.mx_quantize(x, 32)
        assert sb[0, 0] == 127 + k
    # the block maximum never saturates by more than the (448, 512) window
    x = np.zeros((1, 32)); x[0, 0] = hi
    codes, sb = mx.mx_quantize(x, 32)
    assert codes[0, 0] == 0x7E


def test_nonfinite_block():
    x = np.zeros((2, 32))
    x[0, 5] = np.nan
    x[1, 9] = np.inf
    codes, sb = mx.mx_quantize(x, 32)
    assert list(sb[:, 0]) == [0xFF, 0xFF]
    assert np.all(codes == 0x7F)


def test_roundtrip_error_bound():
    # after scaling, each normal element is within half a mantissa step (relative 2^-4)
    rng = np.random.default_rng(1)
    x = torch.tensor(rng.standard_normal((64, 128)) * np.exp(rng.standard_normal((64, 1)) * 3),
                     dtype=torch.float32).to(torch.bfloat16).double().numpy()
    codes, sb = mx.mx_quantize(x, 32)
    d = mx.mx_dequantize(codes, sb, 32)
    scale = mx.e8m0_decode(sb)
    scale_el = np.repeat(scale, 32, axis=1)
    y = x / scale_el
    err = np.abs(d - x) / scale_el
    normal = (np.abs(y) >= 2.0 ** -6) & (np.abs(y) <= 448.0)
    assert np.all(err[normal] <= np.abs(y[normal]) * 2.0 ** -4)
    assert np.all(err[np.abs(y) < 2.0 ** -6] <= 2.0 ** -10)
    sat = np.abs(y) > 448.0            # saturated block maxima: clamped to 448
    assert np.all(err[sat] == np.abs(y[sat]) - 448.0)
    # the per-block maximum lands in [256, 448] after scaling
    amax_scaled = np.max(np.abs(y).reshape(64, 4, 32), axis=-1)
    nz = amax_scaled > 0
    assert np.all((amax_scaled[nz] >= 256) & (amax_scaled[nz] < 512))


def test_operand_layouts_and_blocks():
    rng = np.random.default_rng(2)
    B, S, H, D = 1, 96, 2, 128
    v = torch.tensor(rng.standard_normal((B, S, H, D)), dtype=torch.float32).to(torch.bfloat16).double().numpy()
    # rowwise: block = 32 consecutive d of one (b, s, h)
    c, s = mx.quantize_rowwise(v)
    assert c.shape == (B, S, H, D) and s.shape == (B, H, S, D // 32)
    b0 = v[0, 5, 1, 64:96]
    _, sb = mx.mx_quantize(b0[None], 32)
    assert s[0, 1, 5, 2] == sb[0, 0]
    # columnwise: block = 32 consecutive tokens of one (b, h, d); bytes transposed to [B,H,D,S]
    ct, sc = mx.quantize_colwise(v)
    assert ct.shape == (B, H, D, S) and sc.shape == (B, H, D, S // 32)
    col = v[0, 32:64, 1, 7]
    cc, sb = mx.mx_quantize(col[None], 32)
    assert sc[0, 1, 7, 1] == sb[0, 0]
    np.testing.assert_array_equal(ct[0, 1, 7, 32:64], cc[0])
    # token-normalised: one amplitude per (b, s, h) over all D
    cn, sn = mx.quantize_token_norm(v)
    assert cn.shape == (B, S, H, D) and sn.shape == (B, H, S)
    cc, sb = mx.mx_quantize(v[0, 70, 0][None], 128)
    assert sn[0, 0, 70] == sb[0, 0]
    np.testing.assert_array_equal(cn[0, 70, 0], cc[0])
    # decode inverses are consistent with the blocks
    np.testing.assert_array_equal(mx.dequantize_colwise(ct, sc)[0, 32:64, 1, 7],
                                  mx.mx_dequantize(ct[0, 1, 7, 32:64][None], sc[0, 1, 7, 1:2][None], 32)[0])


def test_block_locality():
    # changing one element only changes its own block's bytes and scale
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 128))
    c0, s0 = mx.mx_quantize(x, 32)
    x2 = x.copy(); x2[2, 70] = 1000.0
    c1, s1 = mx.mx_quantize(x2, 32)
    diff_blocks = np.argwhere(s0 != s1)
    assert [tuple(d) for d in diff_blocks] == [(2, 2)]
    mask = np.ones_like(c0, dtype=bool); mask[2, 64:96] = False
    np.testing.assert_array_equal(c0[mask], c1[mask])


# ----------------------------------------------------------------------------------------------
# The "ceil" scale rule (the scale rounded up so that no element saturates).

def test_ceil_rule_worked_example_saturation_block():
    """amax = 3.75: floor rule e = -7 (byte 0x78) saturates 480 to 448 (0x7E); ceil rule e = -6
    (byte 0x79), 3.75 * 64 = 240 = 1.875 * 2^7 exactly, byte 0x77."""
    x = np.array([[3.75] + [0.0] * 31])
    c_f, s_f = mx.mx_quantize(x, 32, "floor")
    c_c, s_c = mx.mx_quantize(x, 32, "ceil")
    assert s_f[0, 0] == 0x78 and c_f[0, 0] == 0x7E
    assert s_c[0, 0] == 0x79 and c_c[0, 0] == 0x77
    assert mx.mx_dequantize(c_c, s_c, 32)[0, 0] == 3.75


def test_ceil_rule_is_the_smallest_non_saturating_scale():
    """Brute force: for random block maxima, e_ceil is the smallest e with amax * 2^-e <= 448, and
    it equals the floor-rule exponent or one more."""
    rng = np.random.default_rng(7)
    amax = np.ldexp(rng.uniform(1.0, 2.0, 4000), rng.integers(-60, 60, 4000))
    amax = np.concatenate([amax, np.ldexp(1.75, np.arange(-20, 20)), np.ldexp(np.nextafter(1.75, 2), np.arange(-20, 20))])
    e = mx.e8m0_exponent(amax, "ceil")
    ef = mx.e8m0_exponent(amax, "floor")
    assert np.all(np.ldexp(amax, -e) <= 448.0)
    assert np.all(np.ldexp(amax, -(e - 1)) > 448.0)
    assert np.all((e == ef) | (e == ef + 1))
    # significand exactly 1.75 keeps the floor exponent (amax * 2^-e = 448 exactly)
    at = np.ldexp(1.75, np.arange(-20, 20))
    np.testing.assert_array_equal(mx.e8m0_exponent(at, "ceil"), mx.e8m0_exponent(at, "floor"))


def test_ceil_rule_never_saturates_and_matches_floor_elsewhere():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((64, 128)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    cc, sc = mx.mx_quantize(x, 32, "ceil")
    cf, sf = mx.mx_quantize(x, 32, "floor")
    dec = mx.mx_dequantize(cc, sc, 32)
    # no element at the saturation code unless it is exactly 448 * 2^e
    y = np.ldexp(x.reshape(64, 4, 32), -(sc.astype(np.int64) - 127)[..., None]).reshape(64, 128)
    assert np.all(np.abs(y) <= 448.0)
    same = (sc == sf)
    np.testing.assert_array_equal(cc.reshape(64, 4, 32)[same], cf.reshape(64, 4, 32)[same])
    assert np.all(np.abs(dec - x) <= np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(x), 1e-300))) - 4).astype(np.int64))
                  + np.ldexp(1.0, (sc.astype(np.int64) - 127 - 10)).repeat(32, axis=1))
