"""Sequences whose length is a multiple of 32 but not of 128 (a partial last 128-token tile).

The quantisers must give the oracle's bytes and scales for every token, and write 0 into the
scale-atom bytes of the last tile that belong to no token.  The attention forward must match the
oracle on every row (tolerances as in test_attn_gpu.py) and write nothing past S.
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

TAIL_S = [32, 96, 160, 224, 416]


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


@pytest.mark.parametrize("S", TAIL_S)
@pytest.mark.parametrize("layout,B,H", [(I.BSHD, 1, 3), (I.SBHD, 2, 2)])
def test_quant_tails(ops, S, layout, B, H):
    w = I.Workload("tail", B, S, H, H, layout=layout, v_pattern="every7x16")
    q, _, v = I.make_qkv(w, seed_offset=40)
    # rowwise
    xq, xsc = ops.mxfp8_quantize_qk_rowwise(q.cuda(), layout)
    torch.cuda.synchronize()
    assert tuple(xsc.shape) == (B, H, S, 4)
    oq, osc = mx.quantize_rowwise(bshd_np(q, layout).astype(np.float64))
    np.testing.assert_array_equal(xsc.cpu().numpy(), osc)
    np.testing.assert_array_equal(bshd_np(xq, layout), oq)
    # columnwise + token-normalised V
    vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize_v_fused(v.cuda(), layout)
    torch.cuda.synchronize()
    vb = bshd_np(v, layout).astype(np.float64)
    assert tuple(vsc.shape) == (B, H, S // 32, 128)
    oc, ocs = mx.quantize_colwise(vb)
    np.testing.assert_array_equal(vsc_as_oracle(vsc.cpu().numpy()), ocs)
    np.testing.assert_array_equal(vt.cpu().numpy(), oc)
    on, onsc = mx.quantize_token_norm(vb)
    np.testing.assert_array_equal(vtn_sc.cpu().numpy(), onsc)
    np.testing.assert_array_equal(bshd_np(vtn, layout), on)


def _oracle_full(w, q, k, v, vt_is_vc=False):
    qb, kb, vb = (bshd_np(t, w.layout).astype(np.float64) for t in (q, k, v))
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb))
    vc = mx.dequantize_colwise(*mx.quantize_colwise(vb))
    vt = vc if vt_is_vc else mx.dequantize_token_norm(*mx.quantize_token_norm(vb))
    return A.causal_attention(qh, kh, vc, vt, w.scale)


@pytest.mark.parametrize("S", TAIL_S)
@pytest.mark.parametrize("layout,B,Hq,Hkv", [(I.BSHD, 1, 4, 2), (I.SBHD, 2, 2, 1)])
@pytest.mark.parametrize("p_terms", [1, 2])
def test_attn_tails(ops, S, layout, B, Hq, Hkv, p_terms):
    w = I.Workload("tail", B, S, Hq, Hkv, layout=layout)
    q, k, v = I.make_qkv(w, seed_offset=50)
    # sentinel-filled outputs one tile longer than S: nothing past S may be written
    Sp = ((S + 127) // 128) * 128
    if layout == I.BSHD:
        o_big = torch.full((B, Sp, Hq, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        o = o_big[:, :S]
    else:
        o_big = torch.full((Sp, B, Hq, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        o = o_big[:S]
    lse_big = torch.full((B * Hq * S + 64,), 3.0, dtype=torch.float32, device="cuda")
    lse = lse_big[: B * Hq * S].view(B, Hq, S)
    ops.forward(q.cuda(), k.cuda(), v.cuda(), layout, w.scale, p_terms=p_terms, o=o, lse=lse)
    torch.cuda.synchronize()
    tail = o_big[:, S:] if layout == I.BSHD else o_big[S:]
    assert bool((tail == 7.0).all()), "O written past S"
    assert bool((lse_big[B * Hq * S:] == 3.0).all()), "LSE written past S"
    Og = bshd_np(o, layout).astype(np.float64)
    Lg = lse.cpu().numpy().astype(np.float64)
    O, L = _oracle_full(w, q, k, v)
    print(S, _compare(Og, Lg, O, L))


@pytest.mark.parametrize("S", [96, 160])
def test_attn_tails_leaky(ops, S):
    w = I.Workload("tail", 1, S, 2, 2)
    q, k, v = I.make_qkv(w, seed_offset=60)
    o, lse = ops.forward(q.cuda(), k.cuda(), v.cuda(), w.layout, w.scale, p_terms=2, leaky=1)
    torch.cuda.synchronize()
    O, L = _oracle_full(w, q, k, v, vt_is_vc=True)
    print(S, _compare(bshd_np(o, w.layout).astype(np.float64), lse.cpu().numpy().astype(np.float64), O, L))
