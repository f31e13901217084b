"""Causality on the GPU where every ring and tile boundary is exercised, the scope of the guarantee
for non-finite V, and peaky rows.

PR #3865 page, Description: output row i, and its gradients, never depend on a token after i.
  * Forward: perturbing every token after i (its q, k and v; the V amax of i's own 32-token block
    raised 1000x, later blocks x64) leaves rows <= i bit-identical: O, LSE, and the MXFP8 O bytes
    and scales.  S = 1312 = 10 x 128 + 32, so the four-stage K/V ring wraps twice and the last key
    tile is partial; GQA 16/4 in BSHD (B=1) and SBHD (B=2); one and two E4M3 terms for P.
  * Backward: tokens after i change -> dQ of rows <= i bit-identical; queries and dO before i
    change -> dK and dV of tokens >= i bit-identical (O and LSE recomputed by the forward each time).
  * Non-finite V: the diagonal tile's MMAs multiply the zero weights of keys after a row with
    those keys' V, and 0 x NaN is NaN, so inside the 128-token tile of a non-finite V token the
    earlier rows are not covered (the header states V must be finite).  Rows of earlier tiles stay
    bit-identical, which this test pins.
  * Peaky rows: one dominant key and thousands of keys 12-16 (log2) below it, then a later key 10
    above it (a rescale).  The small weights must survive the E4M3 P: each 32-key block carries its
    own scale, so they are not flushed; O must match the oracle within the tolerances.
"""
import math

import numpy as np
import pytest
import torch

from block_scaled_causal_gb300 import inputs as I
from oracle import attention as A
from oracle import mx
from tests.test_attn_gpu import _compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def _bits(x):
    x = x.contiguous()
    return x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32) if x.dtype == torch.float32 else x


def _perturb_after(q, k, v, i, layout, do=None):
    """Copies (in `layout`) with every token after i changed."""
    out = [t.clone() for t in (q, k, v)] + ([do.clone()] if do is not None else [])
    qb, kb, vb = (I.to_bshd(t, layout) for t in out[:3])
    S = qb.shape[1]
    g = torch.Generator().manual_seed(1000 + i)
    qb[:, i + 1:] = torch.randn(qb[:, i + 1:].shape, generator=g).to(torch.bfloat16)
    kb[:, i + 1:] = -3.0 * kb[:, i + 1:]
    vb[:, i + 1:] = vb[:, i + 1:] + 5.0
    last = 32 * (i // 32) + 31
    if i < last < S:
        vb[:, last] = vb[:, last] * 1000.0            # raises the V amax of i's own 32-block
    if last + 1 < S:
        vb[:, last + 1:] = vb[:, last + 1:] * 64.0
    if do is not None:
        db = I.to_bshd(out[3], layout)
        db[:, i + 1:] = -2.0 * db[:, i + 1:]
    return out


FWD_ROWS = [0, 31, 32, 500, 640, 1023, 1151, 1152, 1279, 1280, 1300, 1311]


@pytest.mark.parametrize("layout,B", [(I.BSHD, 1), (I.SBHD, 2)])
@pytest.mark.parametrize("p_terms", [1, 2])
def test_forward_causality_ring_wraps(ops, layout, B, p_terms):
    w = I.Workload("c", B, 1312, 16, 4, layout=layout)
    q, k, v = I.make_qkv(w, seed_offset=20)

    def run(a, b, c):
        return ops.forward(a.cuda(), b.cuda(), c.cuda(), layout, w.scale, p_terms=p_terms, o8_out=True)

    o0, l0, e0, s0 = run(q, k, v)
    ob0, eb0 = I.to_bshd(o0, layout), I.to_bshd(e0, layout)
    for i in FWD_ROWS:
        o1, l1, e1, s1 = run(*_perturb_after(q, k, v, i, layout))
        torch.cuda.synchronize()
        ob1, eb1 = I.to_bshd(o1, layout), I.to_bshd(e1, layout)
        assert torch.equal(_bits(ob0[:, : i + 1]), _bits(ob1[:, : i + 1])), "O rows <= %d changed" % i
        assert torch.equal(_bits(l0[..., : i + 1]), _bits(l1[..., : i + 1])), "LSE rows <= %d changed" % i
        assert torch.equal(eb0[:, : i + 1].contiguous(), eb1[:, : i + 1].contiguous()), "E4M3 O rows <= %d" % i
        assert torch.equal(s0[:, :, : i + 1].contiguous(), s1[:, :, : i + 1].contiguous()), "O scales rows <= %d" % i
        if i + 1 < w.S:
            assert not torch.equal(_bits(ob0[:, i + 1:]), _bits(ob1[:, i + 1:]))   # later rows did change


BWD_CASES = [(I.BSHD, 1, 416, 8, 2, [31, 255, 383, 384, 400, 415]),
             (I.SBHD, 2, 1312, 16, 4, [100, 640, 1279, 1300])]


@pytest.mark.parametrize("layout,B,S,Hq,Hkv,rows", BWD_CASES)
def test_backward_causality(ops, layout, B, S, Hq, Hkv, rows):
    w = I.Workload("cb", B, S, Hq, Hkv, layout=layout)
    q, k, v, do = I.make_qkv(w, seed_offset=60, with_do=True)

    def fb(a, b, c, d):
        return ops.forward_backward(a.cuda(), b.cuda(), c.cuda(), d.cuda(), layout, w.scale, p_terms=2)

    _, _, dq0, dk0, dv0 = fb(q, k, v, do)
    dqb0, dkb0, dvb0 = (I.to_bshd(t, layout) for t in (dq0, dk0, dv0))
    for i in rows:
        # every token after i changes (q, k, v and dO): dQ of rows <= i is unchanged
        _, _, dq1, _, _ = fb(*_perturb_after(q, k, v, i, layout, do=do))
        torch.cuda.synchronize()
        assert torch.equal(_bits(dqb0[:, : i + 1]), _bits(I.to_bshd(dq1, layout)[:, : i + 1])), "dQ rows <= %d" % i
        # queries and dO before i change: dK and dV of tokens >= i are unchanged
        q3, do3 = q.clone(), do.clone()
        qb, db = I.to_bshd(q3, layout), I.to_bshd(do3, layout)
        qb[:, :i] = (qb[:, :i].float() * 1.5 + 0.25).to(torch.bfloat16)
        db[:, :i] = (db[:, :i].float() * 0.25).to(torch.bfloat16)
        _, _, _, dk3, dv3 = fb(q3, k, v, do3)
        torch.cuda.synchronize()
        assert torch.equal(_bits(dkb0[:, i:]), _bits(I.to_bshd(dk3, layout)[:, i:])), "dK tokens >= %d" % i
        assert torch.equal(_bits(dvb0[:, i:]), _bits(I.to_bshd(dv3, layout)[:, i:])), "dV tokens >= %d" % i
        if i > 0:
            assert not torch.equal(_bits(dkb0[:, :i]), _bits(I.to_bshd(dk3, layout)[:, :i]))


@pytest.mark.parametrize("j,val", [(300, float("nan")), (383, float("inf")), (287, float("-inf"))])
def test_nonfinite_v_earlier_tiles_unchanged(ops, j, val):
    w = I.Workload("nf", 1, 512, 4, 2)
    q, k, v = I.make_qkv(w, seed_offset=70)
    v2 = v.clone()
    v2[:, j, :, 5] = val
    for p_terms in (1, 2):
        o0, l0 = ops.forward(q.cuda(), k.cuda(), v.cuda(), w.layout, w.scale, p_terms=p_terms)
        o1, l1 = ops.forward(q.cuda(), k.cuda(), v2.cuda(), w.layout, w.scale, p_terms=p_terms)
        torch.cuda.synchronize()
        t0 = 128 * (j // 128)        # the first row of the token's 128-token tile
        assert torch.equal(_bits(o0[:, :t0]), _bits(o1[:, :t0])), (j, p_terms)
        assert torch.equal(_bits(l0[..., :t0]), _bits(l1[..., :t0])), (j, p_terms)
        # rows after the token's 32-block read its columnwise block: non-finite there
        assert not torch.isfinite(o1[:, 32 * (j // 32) + 32:].float()).all()


def _peaky_inputs(S, seed):
    """Every query row is c e_0 (plus small noise); key 0 dominates with log2-score Y, keys 1..S-1
    sit 12-16 below it, and key S/2 + 2 sits 10 above it (a rescale).  V ~ N(0, 1)."""
    D = 128
    scale = 1.0 / math.sqrt(D)
    c = 8.0
    unit = scale * math.log2(math.e) * c            # log2-score per unit of k along e_0
    g = torch.Generator().manual_seed(seed)
    Y = 20.0
    y = Y - 12.0 - 4.0 * torch.rand(S, generator=g, dtype=torch.float64)
    y[0] = Y
    y[S // 2 + 2] = Y + 10.0
    q = 0.01 * torch.randn((1, S, 1, D), generator=g, dtype=torch.float64)
    q[..., 0] = c
    k = torch.zeros((1, S, 1, D), dtype=torch.float64)
    k[0, :, 0, 0] = y / unit
    v = torch.randn((1, S, 1, D), generator=g, dtype=torch.float64)
    return tuple(t.to(torch.bfloat16) for t in (q, k, v)), scale


@pytest.mark.parametrize("p_terms", [1, 2])
def test_peaky_rows_keep_small_weights(ops, p_terms):
    S = 4096
    (q, k, v), scale = _peaky_inputs(S, 5)
    o, lse = ops.forward(q.cuda(), k.cuda(), v.cuda(), I.BSHD, scale, p_terms=p_terms)
    torch.cuda.synchronize()
    qb, kb, vb = (t.float().numpy().astype(np.float64) for t in (q, k, v))
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb))
    vc = mx.dequantize_colwise(*mx.quantize_colwise(vb))
    vt = mx.dequantize_token_norm(*mx.quantize_token_norm(vb))
    O, L = A.causal_attention(qh, kh, vc, vt, scale)
    # the band below the dominant key carries real mass: row 2000 (before the rescale key) would be
    # V_0 alone without it, and is more than 0.1 away from that
    assert np.abs(O[0, 2000, 0] - vc[0, 0, 0]).max() > 0.1
    Og = o.cpu().float().numpy().astype(np.float64)
    Lg = lse.cpu().numpy().astype(np.float64)
    print(_compare(Og, Lg, O, L))
