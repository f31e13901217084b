"""MXFP8 O output of the attention forward (E4M3 O, one UE8M0 scale per 32 head-dim elements,
compact [B,Hq,S,D/32] like Q's scales), through the C ABI.

The E4M3 O is the MX quantisation of the kernel's fp32 O, which the test never sees; it sees the
BF16 O of the same call (that fp32 O rounded once) and the fp64 oracle.  So:
  * value check against the oracle: |dec(O8) - O| <= attention tolerance + the E4M3 rounding of
    the element (half a step, or the saturation at 448 * 2^e that the floor scale rule allows);
  * rule check against the call's own BF16 O, exact wherever BF16 rounding cannot have changed
    the outcome: the scale byte is floor(log2 amax) - 8 + 127 of the block, and each byte is the
    oracle's E4M3 round-to-nearest-even of O * 2^-e; cases within BF16 rounding of a power of two
    (scale) or of an E4M3 rounding midpoint (byte) are skipped, and must stay a small minority;
  * asking for BF16 O as well changes no E4M3 byte.
"""
import numpy as np
import pytest
import torch

from block_scaled_causal_gb300 import inputs as I
from oracle import attention as A
from oracle import mx
from tests._helpers import bshd_np

pytestmark = pytest.mark.gpu

ATT_ABS = 3e-2     # attention max-abs tolerance (p_terms=2 path)


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def _bf16_half_ulp(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -126, np.ldexp(1.0, (e - 8).astype(np.int64)), 2.0 ** -134)


def _oracle(w, q, k, v):
    qb, kb, vb = (bshd_np(t, w.layout).astype(np.float64) for t in (q, k, v))
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb))
    vc = mx.dequantize_colwise(*mx.quantize_colwise(vb))
    vt = mx.dequantize_token_norm(*mx.quantize_token_norm(vb))
    return A.causal_attention(qh, kh, vc, vt, w.scale)


def _run(ops, w, q, k, v, bf16_out=True):
    o, lse, o8, osc = ops.forward(q.cuda(), k.cuda(), v.cuda(), w.layout, w.scale, p_terms=2, o8_out=True,
                                  bf16_out=bf16_out)
    torch.cuda.synchronize()
    return o, o8, osc


def _check(w, o, o8, osc, O):
    S = w.S
    codes = bshd_np(o8, w.layout)                                   # [B,S,H,128] bytes
    sc_all = osc.cpu().numpy()                                      # [B,H,S,4]
    assert sc_all.shape[2] == S
    sc = np.ascontiguousarray(sc_all.transpose(0, 2, 1, 3))         # [B,S,H,4]
    e = sc.astype(np.int64) - 127
    dec = mx.mx_dequantize(codes, sc, 32)
    assert np.all(np.isfinite(dec))
    # value check against the oracle
    Ob = O.reshape(O.shape[:-1] + (4, 32))
    eb = e[..., None]
    a = np.abs(Ob)
    half_step = np.maximum(np.ldexp(1.0, (np.floor(np.log2(np.maximum(a, 1e-300))) - 4).astype(np.int64)),
                           np.ldexp(1.0, eb - 10))
    sat = np.maximum(0.0, a + ATT_ABS - 448.0 * np.ldexp(1.0, eb))
    tol = (ATT_ABS + half_step + sat).reshape(O.shape)
    err = np.abs(dec - O)
    assert np.all(err <= tol), "worst excess %.3e" % (err - tol).max()
    # rule check against the call's own BF16 O: the fp32 O lies within half a BF16 ulp of it
    ob = bshd_np(o, w.layout).astype(np.float64).reshape(O.shape[:-1] + (4, 32))
    hu = _bf16_half_ulp(ob)
    amax = np.abs(ob).max(axis=-1)
    hu_amax = _bf16_half_ulp(amax)
    p2 = np.ldexp(1.0, np.round(np.log2(np.maximum(amax, 1e-300))).astype(np.int64))
    near_pow2 = np.abs(amax - p2) <= hu_amax                          # the fp32 amax may sit across 2^k
    e_ref = mx.e8m0_exponent(amax)
    ok_scale = near_pow2 | (e_ref == e)
    assert ok_scale.all(), "scale bytes off the MX rule in %d blocks" % (~ok_scale).sum()
    y = np.ldexp(ob, -eb)                                           # O * 2^-e on the kernel's scale
    hy = np.ldexp(hu, -eb)
    ref_codes = mx.e4m3_encode(mx.e4m3_round(y)).reshape(codes.shape)
    # an E4M3 rounding midpoint (or the 448 saturation edge) within hy of y: the fp32 value may
    # have rounded the other way
    ay = np.abs(y)
    ex = np.where(ay >= 2.0 ** -6, np.floor(np.log2(np.maximum(ay, 1e-300))), -6.0)
    step = np.ldexp(1.0, (ex - 3).astype(np.int64))
    mid = (np.floor(ay / step) + 0.5) * step
    mid_lo = mid - step
    ambiguous = (np.minimum(np.abs(ay - mid), np.abs(ay - mid_lo)) <= hy) | (np.abs(ay - 448.0) <= hy + 16.0) \
        | near_pow2[..., None]
    ambiguous = ambiguous.reshape(codes.shape)
    bad = (ref_codes != codes) & ~ambiguous
    assert not bad.any(), "%d E4M3 bytes off the rule" % bad.sum()
    assert ambiguous.mean() < 0.10, "too many ambiguous elements: %.3f" % ambiguous.mean()
    return err.max(), ambiguous.mean()


CASES = [("tiny_s128_h2_every7x16", None), ("g", I.Workload("g", 1, 256, 4, 2, layout=I.BSHD)),
         ("s", I.Workload("s", 2, 384, 2, 2, layout=I.SBHD)), ("tail", I.Workload("tail", 1, 160, 4, 2)),
         ("gqa_s8k_h16_kv4", None)]


@pytest.mark.parametrize("name,w", CASES)
def test_o8_against_oracle(ops, name, w):
    w = I.WORKLOADS[name] if w is None else w
    q, k, v = I.make_qkv(w, seed_offset=70)
    o, o8, osc = _run(ops, w, q, k, v)
    O, _ = _oracle(w, q, k, v)
    print(name, "max |dec - O| %.3e, ambiguous %.4f" % _check(w, o, o8, osc, O))


def test_o8_only_matches_both(ops):
    w = I.Workload("g", 1, 256, 4, 2)
    q, k, v = I.make_qkv(w, seed_offset=71)
    o, o8a, osca = _run(ops, w, q, k, v, bf16_out=True)
    none, o8b, oscb = _run(ops, w, q, k, v, bf16_out=False)
    assert none is None
    assert torch.equal(o8a, o8b) and torch.equal(osca, oscb)
