"""C-ABI behaviour on the GPU: error statuses launch nothing, non-default streams, CUDA-graph
capture and replay, sentinel-filled outputs fully overwritten with guard bands untouched,
repeatability, and the bounded device-side waits (a wait on a barrier nothing arrives on ends with
a status the host reads, and the context stays usable)."""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_causal_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def _quantised(ops, w, seed=0):
    q, k, v = (t.cuda() for t in I.make_qkv(w, seed_offset=seed))
    qq, qs = ops.mxfp8_quantize_qk_rowwise(q, w.layout)
    kq, ks = ops.mxfp8_quantize_qk_rowwise(k, w.layout)
    vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize_v_fused(v, w.layout)
    return (qq, qs, kq, ks, vt, vsc, vtn, vtn_sc), (q, k, v)


def test_nondefault_stream_and_repeatability(ops):
    w = I.Workload("s", 1, 512, 4, 2)
    q, k, v = (t.cuda() for t in I.make_qkv(w))
    o_ref, l_ref = ops.forward(q, k, v, w.layout, w.scale)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = ops.forward(q, k, v, w.layout, w.scale, stream=s)
    s.synchronize()
    assert torch.equal(o_ref.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l_ref.view(torch.int32), l1.view(torch.int32))


def test_cuda_graph_capture_replay(ops):
    w = I.Workload("g", 1, 512, 4, 2)
    q, k, v = (t.cuda() for t in I.make_qkv(w))
    o_ref, l_ref = ops.forward(q, k, v, w.layout, w.scale)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.forward(q, k, v, w.layout, w.scale, stream=s)      # warm-up outside capture
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            o, l = ops.forward(q, k, v, w.layout, w.scale, stream=s)
    torch.cuda.synchronize()
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_ref.view(torch.int16), o.view(torch.int16))
    assert torch.equal(l_ref.view(torch.int32), l.view(torch.int32))


def test_sentinels_overwritten_and_guards_untouched(ops):
    w = I.Workload("x", 1, 384, 4, 2)
    args, _ = _quantised(ops, w)
    B, S, Hq, D = 1, 384, 4, 128
    n = B * S * Hq * D
    pad = 4096
    obuf = torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * Hq * S + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
    o = obuf[pad:pad + n].view(B, S, Hq, D)
    lse = lbuf[pad:pad + B * Hq * S].view(B, Hq, S)
    ops.mxfp8_causal_attn_fwd(*args, layout=w.layout, softmax_scale=w.scale, o=o, lse=lse)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    assert torch.isnan(obuf[:pad]).all() and torch.isnan(obuf[pad + n:]).all()
    assert torch.isnan(lbuf[:pad]).all() and torch.isnan(lbuf[pad + B * Hq * S:]).all()


def test_errors_launch_nothing(ops):
    w = I.Workload("e", 1, 256, 4, 2)
    args, _ = _quantised(ops, w)
    o = torch.full((1, 256, 4, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 4, 256), 7.0, dtype=torch.float32, device="cuda")
    p = ops.make_attn_params(*args, o, lse, w.layout, w.scale, p_terms=5)
    assert ops.lib.mxfp8_causal_attn_fwd(ctypes.byref(p), None) == 4
    p = ops.make_attn_params(*args, o, lse, w.layout, w.scale)
    p.Hkv = 3
    assert ops.lib.mxfp8_causal_attn_fwd(ctypes.byref(p), None) == 2
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
    with pytest.raises(ops.BscError):
        ops.mxfp8_causal_attn_fwd(*args, layout=w.layout, p_terms=0, o=o, lse=lse)


@pytest.mark.parametrize("S", [128, 640])
@pytest.mark.parametrize("p_terms", [1, 2])   # one softmax set; two sets taking alternate key tiles
def test_bounded_wait_reports_timeout_and_context_survives(ops, S, p_terms):
    w = I.Workload("t", 1, S, 1, 1)
    args, _ = _quantised(ops, w)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    ops.mxfp8_causal_attn_fwd(*args, layout=w.layout, softmax_scale=w.scale, p_terms=p_terms, dev_status=status,
                              wait_timeout_ms=200, debug_stall=1)
    assert ops.bsc_read_device_status(status) == ops.BSC_ERR_DEVICE_TIMEOUT
    assert int(status[0].item()) & 0x100
    # the context is still usable and a normal call gives a normal status
    status.zero_()
    o, lse = ops.mxfp8_causal_attn_fwd(*args, layout=w.layout, softmax_scale=w.scale, p_terms=p_terms,
                                       dev_status=status)
    assert ops.bsc_read_device_status(status) == ops.BSC_OK
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("layout,B,S", [(I.BSHD, 1, 416), (I.SBHD, 2, 160)])
def test_attention_on_oracle_quantised_compact_operands(ops, layout, B, S):
    """The C ABI's operand layouts as documented: E4M3 bytes in the input's layout, compact rowwise
    scales [B,H,S,D/32], V bytes transposed to [B,H,D,S] in natural token order with scales
    [B,H,S/32,D], token-normalised bytes in the input's layout with amplitudes [B,H,S].  Operands
    built by the oracle's quantisers (not the library's) give bit-for-bit the output of the whole
    path on the bf16 inputs, and match the oracle's attention within the tolerances."""
    from oracle import attention as A
    from oracle import mx
    from tests._helpers import bshd_np
    from tests.test_attn_gpu import _compare
    w = I.Workload("x", B, S, 4, 2, layout=layout, v_pattern="every7x16")
    q, k, v = I.make_qkv(w, seed_offset=90)
    qb, kb, vb = (bshd_np(t, layout).astype(np.float64) for t in (q, k, v))
    q8, qsc = mx.quantize_rowwise(qb)
    k8, ksc = mx.quantize_rowwise(kb)
    vt, vsc = mx.quantize_colwise(vb)                       # [B,H,D,S], [B,H,D,S/32]
    vtn, vtn_sc = mx.quantize_token_norm(vb)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    lay = lambda a: I.to_layout(torch.from_numpy(np.ascontiguousarray(a)), layout).cuda()
    ops_in = (lay(q8), dev(qsc), lay(k8), dev(ksc), dev(vt), dev(np.swapaxes(vsc, -1, -2)), lay(vtn), dev(vtn_sc))
    o, lse = ops.mxfp8_causal_attn_fwd(*ops_in, layout, w.scale, p_terms=2)
    o_ref, lse_ref = ops.forward(q.cuda(), k.cuda(), v.cuda(), layout, w.scale, p_terms=2)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))
    O, L = A.causal_attention(mx.dequantize_rowwise(q8, qsc), mx.dequantize_rowwise(k8, ksc),
                              mx.dequantize_colwise(vt, vsc), mx.dequantize_token_norm(vtn, vtn_sc), w.scale)
    print(_compare(bshd_np(o, layout).astype(np.float64), lse.cpu().numpy().astype(np.float64), O, L))
