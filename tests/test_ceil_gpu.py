"""The ceil scale rule (e = ceil(log2(amax / 448))) of the quantisers, through mxfp8_quantize.

Bytes and scales must equal the oracle's under rule="ceil" bit for bit, including blocks whose
maximum sits exactly on, just above, or far above the 1.75 significand where the two rules part,
and blocks whose maximum is subnormal.  The floor rule through the same entry must reproduce the
dedicated calls.  Attention on ceil-quantised operands must match the oracle on the same
operands, with the tolerances of test_attn_gpu.py.
"""
import numpy as np
import pytest
import torch

from block_scaled_causal_gb300 import inputs as I
from oracle import attention as A
from oracle import mx
from tests._helpers import bshd_np, vsc_as_oracle
from tests.test_attn_gpu import _compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def _edge_tensor(B, S, H, layout, seed):
    """Random bf16 values whose 32-element blocks (along D, and along S for V) often have a
    maximum with significand 1.75 (floor = ceil), 1.7578125 (the next bf16: ceil = floor + 1),
    1.9921875, or 1.0, at exponents from subnormal to 2^100."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, S, H, 128), generator=g) * 0.5
    sig = torch.tensor([1.75, 1.7578125, 1.9921875, 1.0, 1.5])
    ex = torch.tensor([-133.0, -127.0, -120.0, -6.0, 0.0, 1.0, 7.0, 8.0, 9.0, 100.0])
    n = B * S * H * 4
    picks = torch.randint(0, 5, (n,), generator=g)
    epick = torch.randint(0, len(ex), (n,), generator=g)
    amax = sig[picks] * torch.pow(2.0, ex[epick])
    blocks = x.reshape(n, 32)
    blocks = blocks / blocks.abs().amax(dim=1, keepdim=True).clamp_min(1e-30) * amax[:, None] * 0.999
    pos = torch.randint(0, 32, (n,), generator=g)
    sign = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0)
    blocks[torch.arange(n), pos] = amax * sign
    x = blocks.reshape(B, S, H, 128).to(torch.bfloat16)
    return I.to_layout(x, layout)


def _inputs(kind, B, S, H, layout, seed):
    if kind == "edge":
        return _edge_tensor(B, S, H, layout, seed)
    w = I.Workload("ceil", B, S, H, H, layout=layout, v_pattern="every7x16")
    return I.make_qkv(w, seed_offset=seed)[2]


SHAPES = [("rand", 1, 256, 3, I.BSHD), ("rand", 2, 160, 2, I.SBHD), ("edge", 1, 256, 2, I.BSHD),
          ("edge", 2, 96, 2, I.SBHD)]


@pytest.mark.parametrize("src,B,S,H,layout", SHAPES)
def test_ceil_quantisers_bit_exact(ops, src, B, S, H, layout):
    x = _inputs(src, B, S, H, layout, 90)
    xb = bshd_np(x, layout).astype(np.float64)
    xd = x.cuda()
    # rowwise
    e4, sc = ops.mxfp8_quantize(ops.QUANT_ROWWISE, xd, layout, ops.SCALE_CEIL)
    torch.cuda.synchronize()
    oc, osc = mx.quantize_rowwise(xb, rule="ceil")
    np.testing.assert_array_equal(sc.cpu().numpy(), osc)
    np.testing.assert_array_equal(bshd_np(e4, layout), oc)
    # the rule is in effect: some blocks differ from the floor rule
    _, fsc = mx.quantize_rowwise(xb)
    assert (fsc != osc).any()
    # V: fused, and each half on its own
    vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize(ops.QUANT_V_FUSED, xd, layout, ops.SCALE_CEIL)
    vt1, vsc1 = ops.mxfp8_quantize(ops.QUANT_V_COLWISE, xd, layout, ops.SCALE_CEIL)
    vtn1, vtn_sc1 = ops.mxfp8_quantize(ops.QUANT_V_TOKEN_NORM, xd, layout, ops.SCALE_CEIL)
    torch.cuda.synchronize()
    for a, b in ((vt, vt1), (vsc, vsc1), (vtn, vtn1), (vtn_sc, vtn_sc1)):
        assert torch.equal(a, b)
    cc, ccs = mx.quantize_colwise(xb, rule="ceil")
    np.testing.assert_array_equal(vsc_as_oracle(vsc.cpu().numpy()), ccs)
    np.testing.assert_array_equal(vt.cpu().numpy(), cc)
    tn, tns = mx.quantize_token_norm(xb, rule="ceil")
    np.testing.assert_array_equal(vtn_sc.cpu().numpy(), tns)
    np.testing.assert_array_equal(bshd_np(vtn, layout), tn)


def test_floor_through_entry_matches_dedicated_calls(ops):
    x = _edge_tensor(1, 256, 2, I.BSHD, 91).cuda()
    a = ops.mxfp8_quantize(ops.QUANT_ROWWISE, x, I.BSHD, ops.SCALE_FLOOR)
    b = ops.mxfp8_quantize_qk_rowwise(x, I.BSHD)
    c = ops.mxfp8_quantize(ops.QUANT_V_FUSED, x, I.BSHD, ops.SCALE_FLOOR)
    d = ops.mxfp8_quantize_v_fused(x, I.BSHD)
    torch.cuda.synchronize()
    for u, v in zip(a + c, b + tuple(d)):
        assert torch.equal(u, v)


@pytest.mark.parametrize("S,Hq,Hkv,layout,B", [(256, 4, 2, I.BSHD, 1), (160, 2, 1, I.SBHD, 2)])
def test_attn_on_ceil_operands(ops, S, Hq, Hkv, layout, B):
    w = I.Workload("ceil", B, S, Hq, Hkv, layout=layout, v_pattern="every7x16")
    q, k, v = I.make_qkv(w, seed_offset=92)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    qq, qs = ops.mxfp8_quantize(ops.QUANT_ROWWISE, qd, layout, ops.SCALE_CEIL)
    kq, ks = ops.mxfp8_quantize(ops.QUANT_ROWWISE, kd, layout, ops.SCALE_CEIL)
    vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize(ops.QUANT_V_FUSED, vd, layout, ops.SCALE_CEIL)
    o, lse = ops.mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, layout, w.scale, p_terms=2)
    torch.cuda.synchronize()
    qb, kb, vb = (bshd_np(t, layout).astype(np.float64) for t in (q, k, v))
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb, rule="ceil"))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb, rule="ceil"))
    vc = mx.dequantize_colwise(*mx.quantize_colwise(vb, rule="ceil"))
    vtt = mx.dequantize_token_norm(*mx.quantize_token_norm(vb, rule="ceil"))
    O, L = A.causal_attention(qh, kh, vc, vtt, w.scale)
    print(_compare(bshd_np(o, layout).astype(np.float64), lse.cpu().numpy().astype(np.float64), O, L))
