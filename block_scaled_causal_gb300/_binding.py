"""ctypes binding of libbsc.so: argument marshalling only (every step runs in the CUDA library).

The functions keep the C names of include/bsc.h.  Tensors are torch CUDA tensors; outputs are
allocated with torch when not given.  A missing library raises at import time: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

BSHD = 0
SBHD = 1

BSC_OK = 0
BSC_ERR_DEVICE_TIMEOUT = 6


def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError("libbsc.so is not built (%s); run `python -m block_scaled_causal_gb300.build`" % path)
    lib = ctypes.CDLL(path)
    vp, i32, u8p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    lib.bsc_abi_version.restype = i32
    lib.bsc_status_string.restype = ctypes.c_char_p
    lib.bsc_status_string.argtypes = [i32]
    for name in ("mxfp8_quantize_qk_rowwise", "mxfp8_quantize_v_colwise", "v_token_normalize"):
        f = getattr(lib, name)
        f.restype = i32
        f.argtypes = [vp, i32, i32, i32, i32, i32, u8p, u8p, vp]
    lib.mxfp8_quantize_v_fused.restype = i32
    lib.mxfp8_quantize_v_fused.argtypes = [vp, i32, i32, i32, i32, i32, u8p, u8p, u8p, u8p, vp]
    lib.mxfp8_causal_attn_fwd.restype = i32
    lib.mxfp8_causal_attn_fwd.argtypes = [ctypes.POINTER(AttnFwdParams), vp]
    lib.mxfp8_quantize_qkv.restype = i32
    lib.mxfp8_quantize_qkv.argtypes = [ctypes.POINTER(QkvQuantParams), vp]
    lib.mxfp8_quantize.restype = i32
    lib.mxfp8_quantize.argtypes = [ctypes.POINTER(QuantParams), vp]
    lib.bf16_attn_bwd.restype = i32
    lib.bf16_attn_bwd.argtypes = [ctypes.POINTER(AttnBwdParams), vp]
    lib.bf16_attn_bwd_static.restype = i32
    lib.bf16_attn_bwd_static.argtypes = [ctypes.POINTER(AttnBwdParams), vp]
    lib.bf16_attn_bwd_static_capacity.restype = ctypes.c_size_t
    lib.bf16_attn_bwd_static_capacity.argtypes = []
    lib.bf16_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.bf16_attn_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.bsc_read_device_status.restype = i32
    lib.bsc_read_device_status.argtypes = [vp, vp]
    return lib


class AttnFwdParams(ctypes.Structure):
    """Mirror of bsc_attn_fwd_params."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_sc", ctypes.c_void_p),
        ("k", ctypes.c_void_p), ("k_sc", ctypes.c_void_p),
        ("v_t", ctypes.c_void_p), ("v_sc", ctypes.c_void_p),
        ("vtn", ctypes.c_void_p), ("vtn_sc", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("S", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("D", ctypes.c_int), ("layout", ctypes.c_int), ("softmax_scale", ctypes.c_float),
        ("p_terms", ctypes.c_int), ("leaky", ctypes.c_int),
        ("dev_status", ctypes.c_void_p), ("wait_timeout_ms", ctypes.c_uint32),
        ("debug_stall", ctypes.c_int),
        ("o_e4m3", ctypes.c_void_p), ("o_sc", ctypes.c_void_p),
    ]


class QuantParams(ctypes.Structure):
    """Mirror of bsc_quant_params."""
    _fields_ = [
        ("kind", ctypes.c_int), ("x", ctypes.c_void_p),
        ("B", ctypes.c_int), ("S", ctypes.c_int), ("H", ctypes.c_int), ("D", ctypes.c_int),
        ("layout", ctypes.c_int), ("rule", ctypes.c_int),
        ("e4m3", ctypes.c_void_p), ("sc", ctypes.c_void_p),
        ("vtn_e4m3", ctypes.c_void_p), ("vtn_sc", ctypes.c_void_p),
    ]


class QkvQuantParams(ctypes.Structure):
    """Mirror of bsc_qkv_quant_params."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("B", ctypes.c_int), ("S", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("layout", ctypes.c_int), ("rule", ctypes.c_int),
        ("q_e4m3", ctypes.c_void_p), ("q_sc", ctypes.c_void_p), ("k_e4m3", ctypes.c_void_p), ("k_sc", ctypes.c_void_p),
        ("v_e4m3_t", ctypes.c_void_p), ("v_sc", ctypes.c_void_p),
        ("vtn_e4m3", ctypes.c_void_p), ("vtn_sc", ctypes.c_void_p),
    ]


QUANT_ROWWISE, QUANT_V_COLWISE, QUANT_V_TOKEN_NORM, QUANT_V_FUSED = 0, 1, 2, 3
SCALE_FLOOR, SCALE_CEIL = 0, 1


class AttnBwdParams(ctypes.Structure):
    """Mirror of bsc_attn_bwd_params."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_sc", ctypes.c_void_p),
        ("k", ctypes.c_void_p), ("k_sc", ctypes.c_void_p),
        ("vtn", ctypes.c_void_p), ("vtn_sc", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("d_o", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("B", ctypes.c_int), ("S", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("D", ctypes.c_int), ("layout", ctypes.c_int), ("softmax_scale", ctypes.c_float),
        ("dev_status", ctypes.c_void_p), ("wait_timeout_ms", ctypes.c_uint32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


lib = _load()


class BscError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(lib.bsc_status_string(status).decode())
        self.status = status


def _check(status: int):
    if status != BSC_OK:
        raise BscError(status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bshd_dims(x: torch.Tensor, layout: int):
    if x.dim() != 4:
        raise ValueError("expected a 4-D tensor")
    if layout == BSHD:
        B, S, H, D = x.shape
    else:
        S, B, H, D = x.shape
    return B, S, H, D


def _require(x: torch.Tensor, dtype, name):
    if not x.is_cuda or x.dtype != dtype or not x.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))


def mxfp8_quantize_qk_rowwise(x, layout=BSHD, out=None, out_sc=None, stream=None):
    """Returns (E4M3 bytes shaped like x, scales [B, H, S, D/32])."""
    _require(x, torch.bfloat16, "x")
    B, S, H, D = _bshd_dims(x, layout)
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if out is None else out
    out_sc = torch.empty((B, H, S, D // 32), dtype=torch.uint8, device=x.device) if out_sc is None else out_sc
    _check(lib.mxfp8_quantize_qk_rowwise(_ptr(x), B, S, H, D, layout, _ptr(out), _ptr(out_sc), _stream(stream)))
    return out, out_sc


def _v_outputs(v, B, S, H, D, col, tn):
    dev = v.device
    r = []
    if col:
        r += [torch.empty((B, H, D, S), dtype=torch.uint8, device=dev),
              torch.empty((B, H, S // 32, D), dtype=torch.uint8, device=dev)]
    if tn:
        r += [torch.empty(v.shape, dtype=torch.uint8, device=dev),
              torch.empty((B, H, S), dtype=torch.uint8, device=dev)]
    return r


def mxfp8_quantize_v_colwise(v, layout=BSHD, stream=None):
    """Returns (E4M3 bytes of V transposed [B, H, D, S], scales [B, H, S/32, D])."""
    _require(v, torch.bfloat16, "v")
    B, S, H, D = _bshd_dims(v, layout)
    vt, vsc = _v_outputs(v, B, S, H, D, True, False)
    _check(lib.mxfp8_quantize_v_colwise(_ptr(v), B, S, H, D, layout, _ptr(vt), _ptr(vsc), _stream(stream)))
    return vt, vsc


def v_token_normalize(v, layout=BSHD, stream=None):
    """Returns (E4M3 bytes shaped like v, token amplitudes [B, H, S])."""
    _require(v, torch.bfloat16, "v")
    B, S, H, D = _bshd_dims(v, layout)
    vtn, vtn_sc = _v_outputs(v, B, S, H, D, False, True)
    _check(lib.v_token_normalize(_ptr(v), B, S, H, D, layout, _ptr(vtn), _ptr(vtn_sc), _stream(stream)))
    return vtn, vtn_sc


def mxfp8_quantize_v_fused(v, layout=BSHD, out=None, stream=None):
    """Both V quantisations in one pass: (v_t, v_sc, vtn, vtn_sc)."""
    _require(v, torch.bfloat16, "v")
    B, S, H, D = _bshd_dims(v, layout)
    vt, vsc, vtn, vtn_sc = _v_outputs(v, B, S, H, D, True, True) if out is None else out
    _check(lib.mxfp8_quantize_v_fused(_ptr(v), B, S, H, D, layout, _ptr(vt), _ptr(vsc), _ptr(vtn), _ptr(vtn_sc),
                                      _stream(stream)))
    return vt, vsc, vtn, vtn_sc


def make_attn_params(q, q_sc, k, k_sc, v_t, v_sc, vtn, vtn_sc, o, lse, layout, softmax_scale, p_terms=2, leaky=0,
                     dev_status=None, wait_timeout_ms=0, debug_stall=0, o8=None, o_sc=None):
    B, S, Hq, D = _bshd_dims(q, layout)
    Hkv = _bshd_dims(k, layout)[2]
    return AttnFwdParams(q=q.data_ptr(), q_sc=q_sc.data_ptr(), k=k.data_ptr(), k_sc=k_sc.data_ptr(),
                         v_t=v_t.data_ptr(), v_sc=v_sc.data_ptr(),
                         vtn=0 if vtn is None else vtn.data_ptr(), vtn_sc=0 if vtn_sc is None else vtn_sc.data_ptr(),
                         o=0 if o is None else o.data_ptr(), lse=lse.data_ptr(), B=B, S=S, Hq=Hq, Hkv=Hkv, D=D,
                         layout=layout, softmax_scale=softmax_scale, p_terms=p_terms, leaky=leaky,
                         dev_status=0 if dev_status is None else dev_status.data_ptr(),
                         wait_timeout_ms=wait_timeout_ms, debug_stall=debug_stall,
                         o_e4m3=0 if o8 is None else o8.data_ptr(), o_sc=0 if o_sc is None else o_sc.data_ptr())


def mxfp8_causal_attn_fwd(q, q_sc, k, k_sc, v_t, v_sc, vtn, vtn_sc, layout=BSHD, softmax_scale=None, p_terms=2,
                          leaky=0, o=None, lse=None, dev_status=None, wait_timeout_ms=0, debug_stall=0,
                          stream=None, o8_out=False, bf16_out=True, o8=None, o_sc=None):
    """Leak-free causal MXFP8 attention forward on quantised operands.

    Returns (O bf16, LSE fp32); with o8_out=True, (O bf16 or None, LSE, O E4M3 bytes laid out like
    q, O scales [B, Hq, S, D/32]).  p_terms: E4M3 terms of P for the completed blocks (2: the
    tolerance-preserving default; 1: faster, one E4M3 rounding of P).
    """
    B, S, Hq, D = _bshd_dims(q, layout)
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    if bf16_out:
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device) if o is None else o
    else:
        o = None
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device) if lse is None else lse
    if o8_out:
        o8 = torch.empty(q.shape, dtype=torch.uint8, device=q.device) if o8 is None else o8
        o_sc = torch.empty((B, Hq, S, D // 32), dtype=torch.uint8, device=q.device) if o_sc is None else o_sc
    else:
        o8 = o_sc = None
    p = make_attn_params(q, q_sc, k, k_sc, v_t, v_sc, vtn, vtn_sc, o, lse, layout, softmax_scale, p_terms, leaky,
                         dev_status, wait_timeout_ms, debug_stall, o8, o_sc)
    _check(lib.mxfp8_causal_attn_fwd(ctypes.byref(p), _stream(stream)))
    return (o, lse, o8, o_sc) if o8_out else (o, lse)


def bsc_read_device_status(dev_status, stream=None):
    """Synchronises the stream; returns the library status for the device status word."""
    return lib.bsc_read_device_status(_ptr(dev_status), _stream(stream))


def forward(q, k, v, layout=BSHD, softmax_scale=None, p_terms=2, leaky=0, o=None, lse=None, stream=None,
            o8_out=False, bf16_out=True):
    """The whole hot path on bf16 inputs: quantise Q, K rowwise, V columnwise + token-normalised,
    then the leak-free causal attention forward.  Returns (O bf16, LSE fp32); `o` and `lse` may be
    given (laid out like q and [B, Hq, S]).  With o8_out=True the MXFP8 O is returned as well, as
    in mxfp8_causal_attn_fwd."""
    qq, qs, kq, ks, vt, vsc, vtn, vtn_sc = mxfp8_quantize_qkv(q, k, v, layout, token_norm=not leaky, stream=stream)
    return mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, layout, softmax_scale, p_terms, leaky,
                                 o=o, lse=lse, stream=stream, o8_out=o8_out, bf16_out=bf16_out)


def bf16_attn_bwd_workspace_bytes(B, S, Hq, Hkv):
    """Bytes of scratch the backward needs (the C call of the same name)."""
    return int(lib.bf16_attn_bwd_workspace_bytes(B, S, Hq, Hkv))


def _bwd_params(q, q_sc, k, k_sc, vtn, vtn_sc, o, lse, do, layout, softmax_scale, dq, dk, dv, dev_status,
                wait_timeout_ms, workspace):
    B, S, Hq, D = _bshd_dims(q, layout)
    Hkv = _bshd_dims(k, layout)[2]
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    _require(do, torch.bfloat16, "do")
    _require(o, torch.bfloat16, "o")
    dq = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.bfloat16, device=q.device) if dk is None else dk
    dv = torch.empty(k.shape, dtype=torch.bfloat16, device=q.device) if dv is None else dv
    p = AttnBwdParams(q=q.data_ptr(), q_sc=q_sc.data_ptr(), k=k.data_ptr(), k_sc=k_sc.data_ptr(),
                      vtn=vtn.data_ptr(), vtn_sc=vtn_sc.data_ptr(), o=o.data_ptr(), lse=lse.data_ptr(),
                      d_o=do.data_ptr(), dq=dq.data_ptr(), dk=dk.data_ptr(), dv=dv.data_ptr(), B=B, S=S, Hq=Hq,
                      Hkv=Hkv, D=D, layout=layout, softmax_scale=softmax_scale,
                      dev_status=0 if dev_status is None else dev_status.data_ptr(), wait_timeout_ms=wait_timeout_ms,
                      workspace=0 if workspace is None else workspace.data_ptr(),
                      workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size())
    return p, dq, dk, dv


def bf16_attn_bwd(q, q_sc, k, k_sc, vtn, vtn_sc, o, lse, do, layout=BSHD, softmax_scale=None, dq=None, dk=None,
                  dv=None, dev_status=None, wait_timeout_ms=0, stream=None, workspace=None):
    """Backward on decoded operands (quantised Q, K and token-normalised V, the forward's O, LSE);
    returns (dQ, dK, dV) in bf16, laid out like q and k.  `workspace`: a device tensor of at least
    bf16_attn_bwd_workspace_bytes(B, S, Hq, Hkv) bytes, else one is allocated here."""
    if workspace is None:
        B, S, Hq, _ = _bshd_dims(q, layout)
        ws_bytes = bf16_attn_bwd_workspace_bytes(B, S, Hq, _bshd_dims(k, layout)[2])
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    p, dq, dk, dv = _bwd_params(q, q_sc, k, k_sc, vtn, vtn_sc, o, lse, do, layout, softmax_scale, dq, dk, dv,
                                dev_status, wait_timeout_ms, workspace)
    _check(lib.bf16_attn_bwd(ctypes.byref(p), _stream(stream)))
    return dq, dk, dv


def bf16_attn_bwd_static(q, q_sc, k, k_sc, vtn, vtn_sc, o, lse, do, layout=BSHD, softmax_scale=None, dq=None,
                         dk=None, dv=None, dev_status=None, wait_timeout_ms=0, stream=None):
    """bf16_attn_bwd with the library's fixed device workspace (nothing allocated for scratch)."""
    p, dq, dk, dv = _bwd_params(q, q_sc, k, k_sc, vtn, vtn_sc, o, lse, do, layout, softmax_scale, dq, dk, dv,
                                dev_status, wait_timeout_ms, None)
    _check(lib.bf16_attn_bwd_static(ctypes.byref(p), _stream(stream)))
    return dq, dk, dv


def bf16_attn_bwd_static_capacity():
    """Bytes of the fixed workspace bf16_attn_bwd_static uses."""
    return int(lib.bf16_attn_bwd_static_capacity())


def forward_backward(q, k, v, do, layout=BSHD, softmax_scale=None, p_terms=2, stream=None):
    """Forward then the backward on decoded operands; returns (O, LSE, dQ, dK, dV)."""
    qq, qs, kq, ks, vt, vsc, vtn, vtn_sc = mxfp8_quantize_qkv(q, k, v, layout, stream=stream)
    o, lse = mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, layout, softmax_scale, p_terms,
                                   stream=stream)
    dq, dk, dv = bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o, lse, do, layout, softmax_scale, stream=stream)
    return o, lse, dq, dk, dv


def mxfp8_quantize(kind, x, layout=BSHD, rule=SCALE_FLOOR, stream=None):
    """Any quantisation with a chosen scale rule.  Returns the outputs of the matching call:
    (bytes, [B,H,S,D/32] scales) for QUANT_ROWWISE, (V^T bytes, [B,H,S/32,D] scales) for QUANT_V_COLWISE,
    (token-normalised bytes, amplitudes) for QUANT_V_TOKEN_NORM, all four for QUANT_V_FUSED."""
    _require(x, torch.bfloat16, "x")
    B, S, H, D = _bshd_dims(x, layout)
    u8 = dict(dtype=torch.uint8, device=x.device)
    e4m3 = sc = vtn = vtn_sc = None
    if kind == QUANT_ROWWISE:
        e4m3, sc = torch.empty(x.shape, **u8), torch.empty((B, H, S, D // 32), **u8)
    if kind in (QUANT_V_COLWISE, QUANT_V_FUSED):
        e4m3, sc = torch.empty((B, H, D, S), **u8), torch.empty((B, H, S // 32, D), **u8)
    if kind in (QUANT_V_TOKEN_NORM, QUANT_V_FUSED):
        vtn, vtn_sc = torch.empty(x.shape, **u8), torch.empty((B, H, S), **u8)
    p = QuantParams(kind=kind, x=x.data_ptr(), B=B, S=S, H=H, D=D, layout=layout, rule=rule,
                    e4m3=_ptr(e4m3), sc=_ptr(sc), vtn_e4m3=_ptr(vtn), vtn_sc=_ptr(vtn_sc))
    _check(lib.mxfp8_quantize(ctypes.byref(p), _stream(stream)))
    if kind == QUANT_V_FUSED:
        return e4m3, sc, vtn, vtn_sc
    if kind == QUANT_V_TOKEN_NORM:
        return vtn, vtn_sc
    return e4m3, sc


def mxfp8_quantize_qkv(q, k, v, layout=BSHD, rule=SCALE_FLOOR, token_norm=True, out=None, stream=None):
    """Q and K rowwise and V columnwise (+ token-normalised unless token_norm=False) in one launch.
    Returns (q_e4m3, q_sc, k_e4m3, k_sc, v_e4m3_t, v_sc, vtn_e4m3, vtn_sc), the last two None when
    token_norm=False; `out` may give all eight (the last two may be None)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, torch.bfloat16, n)
    B, S, Hq, D = _bshd_dims(q, layout)
    Hkv = _bshd_dims(k, layout)[2]
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("k and v must have the same shape")
    if out is None:
        u8 = dict(dtype=torch.uint8, device=q.device)
        out = (torch.empty(q.shape, **u8), torch.empty((B, Hq, S, D // 32), **u8),
               torch.empty(k.shape, **u8), torch.empty((B, Hkv, S, D // 32), **u8),
               torch.empty((B, Hkv, D, S), **u8), torch.empty((B, Hkv, S // 32, D), **u8),
               torch.empty(v.shape, **u8) if token_norm else None,
               torch.empty((B, Hkv, S), **u8) if token_norm else None)
    qq, qs, kq, ks, vt, vsc, vtn, vtn_sc = out
    p = QkvQuantParams(q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(), B=B, S=S, Hq=Hq, Hkv=Hkv, D=D, layout=layout,
                       rule=rule, q_e4m3=_ptr(qq), q_sc=_ptr(qs), k_e4m3=_ptr(kq), k_sc=_ptr(ks), v_e4m3_t=_ptr(vt),
                       v_sc=_ptr(vsc), vtn_e4m3=_ptr(vtn), vtn_sc=_ptr(vtn_sc))
    _check(lib.mxfp8_quantize_qkv(ctypes.byref(p), _stream(stream)))
    return qq, qs, kq, ks, vt, vsc, vtn, vtn_sc
