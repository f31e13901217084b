"""Q, K and V quantised in one launch (mxfp8_quantize_qkv), through the C ABI.

Its outputs must be byte-identical to the dedicated calls (themselves bit-exact against the
oracle in test_quant_gpu.py, test_tails_gpu.py and test_ceil_gpu.py), under both scale rules, for
GQA and MHA, both layouts and partial last tiles; one case is also compared with the oracle
directly.  With token_norm=False the token-normalised outputs are not produced and the rest is
unchanged.
"""
import numpy as np
import pytest
import torch

from block_scaled_causal_gb300 import inputs as I
from oracle import mx
from tests._helpers import bshd_np, vsc_as_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def _separate(ops, q, k, v, layout, rule):
    qq, qs = ops.mxfp8_quantize(ops.QUANT_ROWWISE, q, layout, rule)
    kq, ks = ops.mxfp8_quantize(ops.QUANT_ROWWISE, k, layout, rule)
    vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize(ops.QUANT_V_FUSED, v, layout, rule)
    return qq, qs, kq, ks, vt, vsc, vtn, vtn_sc


@pytest.mark.parametrize("B,S,Hq,Hkv,layout", [(1, 256, 4, 2, I.BSHD), (2, 160, 2, 2, I.SBHD),
                                               (1, 416, 6, 2, I.BSHD), (1, 32, 1, 1, I.BSHD)])
@pytest.mark.parametrize("rule", [0, 1])
def test_qkv_matches_separate_calls(ops, B, S, Hq, Hkv, layout, rule):
    w = I.Workload("qkv", B, S, Hq, Hkv, layout=layout, v_pattern="every7x16")
    q, k, v = (t.cuda() for t in I.make_qkv(w, seed_offset=100))
    fused = ops.mxfp8_quantize_qkv(q, k, v, layout, rule)
    ref = _separate(ops, q, k, v, layout, rule)
    torch.cuda.synchronize()
    names = ("q_e4m3", "q_sc", "k_e4m3", "k_sc", "v_e4m3_t", "v_sc", "vtn_e4m3", "vtn_sc")
    for name, a, b in zip(names, fused, ref):
        assert torch.equal(a, b), name


def test_qkv_against_oracle(ops):
    w = I.Workload("qkv", 1, 224, 4, 2, layout=I.BSHD, v_pattern="every7x16")
    q, k, v = I.make_qkv(w, seed_offset=101)
    qq, qs, kq, ks, vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize_qkv(q.cuda(), k.cuda(), v.cuda(), w.layout)
    torch.cuda.synchronize()
    S = w.S
    for x, xq, xs in ((q, qq, qs), (k, kq, ks)):
        oc, osc = mx.quantize_rowwise(bshd_np(x, w.layout).astype(np.float64))
        np.testing.assert_array_equal(xs.cpu().numpy(), osc)
        np.testing.assert_array_equal(bshd_np(xq, w.layout), oc)
    vb = bshd_np(v, w.layout).astype(np.float64)
    cc, ccs = mx.quantize_colwise(vb)
    np.testing.assert_array_equal(vsc_as_oracle(vsc.cpu().numpy()), ccs)
    np.testing.assert_array_equal(vt.cpu().numpy(), cc)
    tn, tns = mx.quantize_token_norm(vb)
    np.testing.assert_array_equal(vtn_sc.cpu().numpy(), tns)
    np.testing.assert_array_equal(bshd_np(vtn, w.layout), tn)


def test_qkv_without_token_norm(ops):
    w = I.Workload("qkv", 1, 256, 4, 2)
    q, k, v = (t.cuda() for t in I.make_qkv(w, seed_offset=102))
    part = ops.mxfp8_quantize_qkv(q, k, v, w.layout, token_norm=False)
    full = ops.mxfp8_quantize_qkv(q, k, v, w.layout)
    torch.cuda.synchronize()
    assert part[6] is None and part[7] is None
    for a, b in zip(part[:6], full[:6]):
        assert torch.equal(a, b)


def test_forward_through_fused_quantiser_matches_separate(ops):
    """forward() quantises with the fused call; the attention output equals the one computed
    from the dedicated quantisers' outputs."""
    w = I.Workload("qkv", 1, 384, 4, 2)
    q, k, v = (t.cuda() for t in I.make_qkv(w, seed_offset=103))
    o1, l1 = ops.forward(q, k, v, w.layout, w.scale)
    ref = _separate(ops, q, k, v, w.layout, 0)
    o2, l2 = ops.mxfp8_causal_attn_fwd(*ref, w.layout, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
