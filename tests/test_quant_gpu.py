"""GPU quantisers against the oracle, bit-exact (bytes and scales), through the C ABI."""
import dataclasses

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


def _check_rowwise(ops, x_cpu, layout, rows=None):
    xq, xsc = ops.mxfp8_quantize_qk_rowwise(x_cpu.cuda(), layout)
    torch.cuda.synchronize()
    xb = bshd_np(x_cpu, layout).astype(np.float64)
    gq = bshd_np(xq, layout)
    gs = xsc.cpu().numpy()
    if rows is not None:                   # the rule is per row: a subset of tokens is the same check
        xb, gq, gs = xb[:, rows], gq[:, rows], gs[:, :, rows]
    oq, os_ = mx.quantize_rowwise(xb)
    np.testing.assert_array_equal(gs, os_)
    np.testing.assert_array_equal(gq, oq)


def _check_v(ops, v_cpu, layout, tokens=None):
    vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize_v_fused(v_cpu.cuda(), layout)
    vt2, vsc2 = ops.mxfp8_quantize_v_colwise(v_cpu.cuda(), layout)
    vtn2, vtn_sc2 = ops.v_token_normalize(v_cpu.cuda(), layout)
    torch.cuda.synchronize()
    for a, b in ((vt, vt2), (vsc, vsc2), (vtn, vtn2), (vtn_sc, vtn_sc2)):
        assert torch.equal(a, b)
    vb = bshd_np(v_cpu, layout).astype(np.float64)
    g_vt = vt.cpu().numpy()
    g_vsc = vsc_as_oracle(vsc.cpu().numpy())
    g_vtn = bshd_np(vtn, layout)
    g_vtn_sc = vtn_sc.cpu().numpy()
    if tokens is not None:                 # whole 128-token tiles
        sl = np.concatenate([np.arange(t * 128, t * 128 + 128) for t in tokens])
        blocks = np.concatenate([np.arange(t * 4, t * 4 + 4) for t in tokens])
        vb, g_vt, g_vsc = vb[:, sl], g_vt[..., sl], g_vsc[..., blocks]
        g_vtn, g_vtn_sc = g_vtn[:, sl], g_vtn_sc[..., sl]
    oc, osc = mx.quantize_colwise(vb)
    np.testing.assert_array_equal(g_vsc, osc)
    np.testing.assert_array_equal(g_vt, oc)
    on, onsc = mx.quantize_token_norm(vb)
    np.testing.assert_array_equal(g_vtn_sc, onsc)
    np.testing.assert_array_equal(g_vtn, on)


SMALL = ["tiny_s128_h2_every7x16", "gqa_s8k_h16_kv4"]


@pytest.mark.parametrize("name", SMALL)
def test_quant_parity_full(ops, name):
    w = I.WORKLOADS[name]
    q, k, v = I.make_qkv(w)
    _check_rowwise(ops, q, w.layout)
    _check_rowwise(ops, k, w.layout)
    _check_v(ops, v, w.layout)


@pytest.mark.parametrize("name", ["mha_s16k_h16_heavy1pct", "gqa_s32k_h16_kv4", "mha_b2_s32k_h16_sbhd"])
def test_quant_parity_sampled(ops, name):
    w = I.WORKLOADS[name]
    q, k, v = I.make_qkv(w)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(256), np.arange(w.S - 256, w.S), rng.integers(0, w.S, 512)]))
    _check_rowwise(ops, q, w.layout, rows)
    _check_rowwise(ops, k, w.layout, rows)
    tiles = sorted(set([0, 1, w.S // 128 - 1] + list(rng.integers(0, w.S // 128, 6))))
    _check_v(ops, v, w.layout, tiles)


def _bf16_bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def test_edge_blocks(ops):
    """All-zero blocks, single nonzero, RNE ties, saturation, subnormals, signed zeros, extreme
    magnitudes, NaN and Inf blocks, in both quantisation directions."""
    S, H = 256, 2
    x = torch.randn((1, S, H, 128), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    x[0, 0] = 0.0                                      # all-zero rows
    x[0, 1] = 0.0
    x[0, 1, 0, 5] = 3.0                                # a single nonzero
    ties = [3.0, 0.0205078125, 0.0224609375, -0.02001953125, 1.0013580322265625e-4, 1e-8, -1e-8, -0.0]
    x[0, 2, 0, :8] = _bf16_bits(ties)
    x[0, 3, 1, :32] = 3.75                             # saturation of the block maximum
    x[0, 4, 0, :] = _bf16_bits([2.0 ** -130] * 128)    # bf16 subnormals, scale clamps at 2^-127
    x[0, 5, 0, :] = 3.0e38                             # near the top of the range
    x[0, 6, 1, :16] = -0.0
    x[0, 7, 0, 40] = float("nan")                      # a NaN block and an Inf block
    x[0, 8, 1, 100] = float("inf")
    x[0, 40:72, 0, 9] = 0.0                            # an all-zero V column block
    x[0, 64:96, 1, 3] = 2.0 ** -133                    # smallest bf16 subnormal column
    _check_rowwise(ops, x, I.BSHD)
    _check_v(ops, x, I.BSHD)


def test_sbhd_equals_bshd(ops):
    w = dataclasses.replace(I.WORKLOADS["gqa_s8k_h16_kv4"], S=1024, B=3)
    q, _, v = I.make_qkv(w)
    qs = I.to_layout(q, I.SBHD)
    a, asc = ops.mxfp8_quantize_qk_rowwise(q.cuda(), I.BSHD)
    b, bsc = ops.mxfp8_quantize_qk_rowwise(qs.cuda(), I.SBHD)
    assert torch.equal(asc, bsc)
    assert torch.equal(a, b.permute(1, 0, 2, 3))
    _check_v(ops, I.to_layout(v, I.SBHD), I.SBHD)


def test_guard_bands_untouched(ops):
    """Outputs inside larger buffers: bytes outside the written range keep their sentinel."""
    B, S, H = 1, 256, 2
    x = torch.randn((B, S, H, 128), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
    pad = 4096
    n = B * S * H * 128
    buf = torch.full((n + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda")
    sbuf = torch.full((B * H * S * 4 + 2 * pad,), 0x5A, dtype=torch.uint8, device="cuda")
    out = buf[pad:pad + n].view(B, S, H, 128)
    osc = sbuf[pad:pad + B * H * S * 4].view(B, H, S, 4)
    ops.mxfp8_quantize_qk_rowwise(x, I.BSHD, out=out, out_sc=osc)
    torch.cuda.synchronize()
    assert bool((buf[:pad] == 0xA5).all()) and bool((buf[pad + n:] == 0xA5).all())
    assert bool((sbuf[:pad] == 0x5A).all()) and bool((sbuf[pad + B * H * S * 4:] == 0x5A).all())
    ref, rsc = ops.mxfp8_quantize_qk_rowwise(x, I.BSHD)
    assert torch.equal(out, ref) and torch.equal(osc, rsc)
