"""Outputs written into caller buffers that sit inside sentinel-filled allocations with guard bands
on both sides: every output of the fused Q/K/V quantiser (E4M3 bytes and compact scales, both V
forms), the attention's BF16 O, LSE and MXFP8 O bytes and scales, and dQ, dK, dV.  Each must equal
the output of the same call into fresh buffers, and no guard byte may change.  Shapes have a partial
last 128-token tile (S % 128 == 32) in both layouts."""
import math

import pytest
import torch

from block_scaled_causal_gb300 import inputs as I

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


class Guarded:
    """A view of `shape` inside a flat allocation filled with `fill`, GUARD bytes of it each side."""

    def __init__(self, shape, dtype, fill):
        self.n = math.prod(shape)
        self.g = GUARD // torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((self.n + 2 * self.g,), fill, dtype=dtype, device="cuda")
        self.fill = self.buf[:1].clone()
        self.view = self.buf[self.g:self.g + self.n].view(shape)

    def guards_intact(self):
        raw = self.buf.view(torch.uint8) if self.buf.dtype != torch.uint8 else self.buf
        one = self.fill.view(torch.uint8) if self.fill.dtype != torch.uint8 else self.fill
        esz = one.numel()
        pat = one.repeat(self.g)
        return torch.equal(raw[: self.g * esz], pat) and torch.equal(raw[-self.g * esz:], pat)


def _same(a, b):
    a, b = a.contiguous(), b.contiguous()
    if a.dtype in (torch.bfloat16, torch.float32):
        a = a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32)
        b = b.view(a.dtype)
    return torch.equal(a, b)


CASES = [(I.BSHD, 1, 416, 4, 2), (I.SBHD, 2, 160, 2, 1)]


@pytest.mark.parametrize("layout,B,S,Hq,Hkv", CASES)
def test_quantiser_outputs_guarded(ops, layout, B, S, Hq, Hkv):
    w = I.Workload("g", B, S, Hq, Hkv, layout=layout, v_pattern="every7x16")
    q, k, v = (t.cuda() for t in I.make_qkv(w, seed_offset=80))
    ref = ops.mxfp8_quantize_qkv(q, k, v, layout)
    outs = [Guarded(tuple(r.shape), torch.uint8, 0xA5) for r in ref]
    got = ops.mxfp8_quantize_qkv(q, k, v, layout, out=tuple(o.view for o in outs))
    torch.cuda.synchronize()
    for name, r, g, o in zip(("q", "q_sc", "k", "k_sc", "v_t", "v_sc", "vtn", "vtn_sc"), ref, got, outs):
        assert _same(r, g), name
        assert o.guards_intact(), name
    # the fused V quantiser alone, into guarded buffers
    vref = ops.mxfp8_quantize_v_fused(v, layout)
    vouts = [Guarded(tuple(r.shape), torch.uint8, 0x5A) for r in vref]
    vgot = ops.mxfp8_quantize_v_fused(v, layout, out=tuple(o.view for o in vouts))
    torch.cuda.synchronize()
    for r, g, o in zip(vref, vgot, vouts):
        assert _same(r, g) and o.guards_intact()


@pytest.mark.parametrize("layout,B,S,Hq,Hkv", CASES)
@pytest.mark.parametrize("p_terms", [1, 2])
def test_attention_outputs_guarded(ops, layout, B, S, Hq, Hkv, p_terms):
    w = I.Workload("g", B, S, Hq, Hkv, layout=layout)
    q, k, v = (t.cuda() for t in I.make_qkv(w, seed_offset=81))
    quant = ops.mxfp8_quantize_qkv(q, k, v, layout)
    o_r, l_r, e_r, s_r = ops.mxfp8_causal_attn_fwd(*quant, layout, w.scale, p_terms=p_terms, o8_out=True)
    go = Guarded(tuple(o_r.shape), torch.bfloat16, 7.0)
    gl = Guarded(tuple(l_r.shape), torch.float32, 3.0)
    ge = Guarded(tuple(e_r.shape), torch.uint8, 0xA5)
    gs = Guarded(tuple(s_r.shape), torch.uint8, 0x5A)
    ops.mxfp8_causal_attn_fwd(*quant, layout, w.scale, p_terms=p_terms, o8_out=True, o=go.view, lse=gl.view,
                              o8=ge.view, o_sc=gs.view)
    torch.cuda.synchronize()
    for r, g, name in ((o_r, go, "o"), (l_r, gl, "lse"), (e_r, ge, "o_e4m3"), (s_r, gs, "o_sc")):
        assert _same(r, g.view), name
        assert g.guards_intact(), name


@pytest.mark.parametrize("layout,B,S,Hq,Hkv", CASES)
def test_backward_outputs_guarded(ops, layout, B, S, Hq, Hkv):
    w = I.Workload("g", B, S, Hq, Hkv, layout=layout)
    q, k, v, do = (t.cuda() for t in I.make_qkv(w, seed_offset=82, with_do=True))
    qq, qs, kq, ks, vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize_qkv(q, k, v, layout)
    o, lse = ops.mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, layout, w.scale)
    ref = ops.bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o, lse, do, layout, w.scale)
    gq, gk, gv = (Guarded(tuple(r.shape), torch.bfloat16, -5.0) for r in ref)
    ops.bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o, lse, do, layout, w.scale, dq=gq.view, dk=gk.view, dv=gv.view)
    torch.cuda.synchronize()
    for r, g, name in zip(ref, (gq, gk, gv), ("dq", "dk", "dv")):
        assert _same(r, g.view), name
        assert g.guards_intact(), name
