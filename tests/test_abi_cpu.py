"""The C-ABI library loads, exports every function include/bsc.h declares, and rejects bad
arguments with the documented status before touching any device (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsc.h")


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import build
    if not os.path.exists(build.LIB_PATH):
        build.build()
    from block_scaled_causal_gb300 import _binding
    return _binding


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_0-9]+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(ops):
    names = _declared_functions()
    assert {"mxfp8_quantize_qk_rowwise", "mxfp8_quantize_v_colwise", "v_token_normalize",
            "mxfp8_quantize_v_fused", "mxfp8_causal_attn_fwd", "bsc_status_string",
            "bsc_read_device_status", "bsc_abi_version"} <= set(names)
    lib = ctypes.CDLL(ops._build.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(ops):
    for code in range(7):
        assert ops.lib.bsc_status_string(code).decode().startswith("BSC_")
    assert ops.lib.bsc_abi_version() == 3


def test_params_struct_layout(ops):
    # 10 pointers, 5 ints, layout, float, 2 ints, pointer, uint32, int  (x86-64 / aarch64 LP64)
    P = ops.AttnFwdParams
    assert P.B.offset == 80 and P.softmax_scale.offset == 104 and P.dev_status.offset == 120
    assert P.o_e4m3.offset == 136 and P.o_sc.offset == 144
    assert ctypes.sizeof(P) == 152


FAKE = 0x100000   # 16-byte aligned, never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,want", [
    ((FAKE, 1, 128, 2, 64, 0, FAKE, FAKE), 4),       # D != 128
    ((FAKE, 1, 100, 2, 128, 0, FAKE, FAKE), 4),      # S % 32
    ((FAKE, -1, 128, 2, 128, 0, FAKE, FAKE), 2),     # negative size
    ((FAKE, 1, 128, 2, 128, 7, FAKE, FAKE), 2),      # bad layout
    ((None, 1, 128, 2, 128, 0, FAKE, FAKE), 1),      # NULL input
    ((FAKE + 8, 1, 128, 2, 128, 0, FAKE, FAKE), 3),  # misaligned
    ((None, 0, 128, 2, 128, 0, None, None), 0),      # empty problem: nothing to do
])
def test_rowwise_validation(ops, args, want):
    st = ops.lib.mxfp8_quantize_qk_rowwise(*args, None)
    assert st == want


def test_v_validation(ops):
    L = ops.lib
    assert L.mxfp8_quantize_v_fused(FAKE, 1, 128, 2, 128, 0, FAKE, FAKE, None, FAKE, None) == 1
    assert L.mxfp8_quantize_v_colwise(FAKE, 1, 128, 2, 128, 0, FAKE + 4, FAKE, None) == 3
    assert L.v_token_normalize(FAKE, 1, 80, 2, 128, 0, FAKE, FAKE, None) == 4
    assert L.v_token_normalize(FAKE, 2, 0, 2, 128, 1, None, None, None) == 0


def _params(ops, **kw):
    base = dict(q=FAKE, q_sc=FAKE, k=FAKE, k_sc=FAKE, v_t=FAKE, v_sc=FAKE, vtn=FAKE, vtn_sc=FAKE, o=FAKE,
                lse=FAKE, B=1, S=256, Hq=4, Hkv=2, D=128, layout=0, softmax_scale=0.088, p_terms=1, leaky=0,
                dev_status=0, wait_timeout_ms=0, debug_stall=0)
    base.update(kw)
    return ops.AttnFwdParams(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(Hq=3, Hkv=2), 2),
    (dict(Hkv=0), 2),
    (dict(D=64), 4),
    (dict(S=200), 4),
    (dict(p_terms=3), 4),
    (dict(leaky=2), 4),
    (dict(softmax_scale=0.0), 4),                 # the scale must be finite and positive
    (dict(softmax_scale=-0.088), 4),
    (dict(softmax_scale=float("nan")), 4),
    (dict(softmax_scale=float("inf")), 4),
    (dict(layout=2), 2),
    (dict(o=0), 1),
    (dict(vtn=0), 1),
    (dict(lse=FAKE + 4), 3),
    (dict(dev_status=FAKE + 2), 3),
    (dict(S=0), 0),
    (dict(B=0, q=0, k=0), 0),
])
def test_attn_validation(ops, kw, want):
    p = _params(ops, **kw)
    assert ops.lib.mxfp8_causal_attn_fwd(ctypes.byref(p), None) == want


def test_bwd_validation(ops):
    base = dict(q=FAKE, q_sc=FAKE, k=FAKE, k_sc=FAKE, vtn=FAKE, vtn_sc=FAKE, o=FAKE, lse=FAKE, d_o=FAKE, dq=FAKE,
                dk=FAKE, dv=FAKE, B=1, S=256, Hq=4, Hkv=2, D=128, layout=0, softmax_scale=0.088, dev_status=0,
                wait_timeout_ms=0, workspace=FAKE, workspace_bytes=1 << 30)
    for kw, want in ((dict(softmax_scale=-1.0), 4), (dict(softmax_scale=float("nan")), 4), (dict(Hq=3), 2),
                     (dict(dq=0), 1), (dict(dk=FAKE + 8), 3), (dict(S=0), 0), (dict(workspace=0), 1),
                     (dict(workspace=FAKE + 4), 3), (dict(workspace_bytes=256 * (8 * 4 + 256 * 8) - 1), 2)):
        p = ops.AttnBwdParams(**dict(base, **kw))
        assert ops.lib.bf16_attn_bwd(ctypes.byref(p), None) == want, kw
    assert ops.lib.bf16_attn_bwd(None, None) == 1


def test_bwd_workspace_bytes(ops):
    # per padded row: fp32 Dlt and LSE per query row, a 128-element BF16 row per query, key, value
    def want(B, S, Hq, Hkv):
        Sp = -(-S // 128) * 128
        return B * Sp * (8 * Hq + 256 * (Hq + 2 * Hkv))
    for args in ((1, 256, 4, 2), (2, 160, 3, 1), (1, 32768, 16, 4), (2, 32768, 16, 16)):
        assert ops.bf16_attn_bwd_workspace_bytes(*args) == want(*args), args
    assert ops.bf16_attn_bwd_workspace_bytes(0, 256, 4, 2) == 0
    assert ops.bf16_attn_bwd_workspace_bytes(1, 0, 4, 2) == 0
    assert ops.bf16_attn_bwd_workspace_bytes(1, 256, 4, 0) == 0


def test_attn_null_params(ops):
    assert ops.lib.mxfp8_causal_attn_fwd(None, None) == 1
    assert ops.lib.bsc_read_device_status(None, None) == 1


def test_quant_params_struct_layout(ops):
    # int, pointer, 6 ints, 4 pointers (LP64)
    P = ops.QuantParams
    assert P.x.offset == 8 and P.B.offset == 16 and P.rule.offset == 36 and P.e4m3.offset == 40
    assert P.vtn_sc.offset == 64 and ctypes.sizeof(P) == 72


@pytest.mark.parametrize("kw,want", [
    (dict(kind=9), 4),                       # unknown kind
    (dict(rule=2), 4),                       # unknown rule
    (dict(S=100), 4),                        # S % 32
    (dict(layout=5), 2),
    (dict(x=0), 1),
    (dict(sc=FAKE + 1), 3),
    (dict(kind=2, vtn_e4m3=0), 1),           # token-norm needs its own outputs
    (dict(kind=1, e4m3=FAKE + 8), 3),
    (dict(kind=3, S=0), 0),                  # empty problem
    (dict(rule=1, B=0, x=0), 0),
])
def test_quant_entry_validation(ops, kw, want):
    base = dict(kind=0, x=FAKE, B=1, S=128, H=2, D=128, layout=0, rule=1, e4m3=FAKE, sc=FAKE,
                vtn_e4m3=FAKE, vtn_sc=FAKE)
    base.update(kw)
    p = ops.QuantParams(**base)
    assert ops.lib.mxfp8_quantize(ctypes.byref(p), None) == want


def test_quant_entry_null(ops):
    assert ops.lib.mxfp8_quantize(None, None) == 1
    assert ops.lib.mxfp8_quantize_qkv(None, None) == 1


def test_qkv_quant_params_struct_layout(ops):
    P = ops.QkvQuantParams
    assert P.B.offset == 24 and P.rule.offset == 48 and P.q_e4m3.offset == 56 and P.vtn_sc.offset == 112
    assert ctypes.sizeof(P) == 120


@pytest.mark.parametrize("kw,want", [
    (dict(rule=3), 4),
    (dict(Hq=3), 2),                                 # Hq % Hkv
    (dict(Hkv=0), 2),
    (dict(S=96 + 8), 4),
    (dict(layout=4), 2),
    (dict(q=0), 1),
    (dict(vtn_e4m3=0), 1),                           # half a V pair
    (dict(v_e4m3_t=0, v_sc=0, vtn_e4m3=0, vtn_sc=0), 1),   # no V output at all
    (dict(k_sc=FAKE + 4), 3),
    (dict(S=0), 0),
    (dict(B=0, q=0, k=0, v=0), 0),
])
def test_qkv_quant_validation(ops, kw, want):
    base = dict(q=FAKE, k=FAKE, v=FAKE, B=1, S=128, Hq=4, Hkv=2, D=128, layout=0, rule=0, q_e4m3=FAKE, q_sc=FAKE,
                k_e4m3=FAKE, k_sc=FAKE, v_e4m3_t=FAKE, v_sc=FAKE, vtn_e4m3=FAKE, vtn_sc=FAKE)
    base.update(kw)
    p = ops.QkvQuantParams(**base)
    assert ops.lib.mxfp8_quantize_qkv(ctypes.byref(p), None) == want

