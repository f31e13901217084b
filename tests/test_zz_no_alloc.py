"""bf16_attn_bwd_static (the backward with the library's fixed device workspace) against
bf16_attn_bwd with a caller workspace: bit-identical dQ, dK, dV on two consecutive calls (the second
call finds the fixed workspace holding the first call's planes), and refusal of a call larger than
the fixed workspace.  Collected last: the first call of the static form loads the array's module."""
import ctypes

import pytest
import torch

from block_scaled_causal_gb300 import inputs as I


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def test_static_capacity_and_refusal(ops):
    cap = ops.bf16_attn_bwd_static_capacity()
    assert cap == 256 << 20
    # B=2, 16/16, S=32K needs 814 MB: refused before any launch (no device memory is touched)
    need = ops.bf16_attn_bwd_workspace_bytes(2, 32768, 16, 16)
    assert need > cap
    FAKE = 1 << 20
    p = ops.AttnBwdParams(q=FAKE, q_sc=FAKE, k=FAKE, k_sc=FAKE, vtn=FAKE, vtn_sc=FAKE, o=FAKE, lse=FAKE, d_o=FAKE,
                          dq=FAKE, dk=FAKE, dv=FAKE, B=2, S=32768, Hq=16, Hkv=16, D=128, layout=1,
                          softmax_scale=0.088, dev_status=0, wait_timeout_ms=0, workspace=0, workspace_bytes=0)
    assert ops.lib.bf16_attn_bwd_static(ctypes.byref(p), None) == 2   # BSC_ERR_SHAPE
    assert ops.lib.bf16_attn_bwd_static(None, None) == 1


@pytest.mark.gpu
@pytest.mark.parametrize("layout,B,S,Hq,Hkv", [(I.BSHD, 1, 1312, 16, 4), (I.SBHD, 2, 416, 8, 8)])
def test_static_matches_caller_workspace(ops, layout, B, S, Hq, Hkv):
    w = I.Workload("na", B, S, Hq, Hkv, layout=layout)
    outs = []
    for seed in (91, 92):   # two consecutive calls, different inputs
        q, k, v, do = (t.cuda() for t in I.make_qkv(w, seed_offset=seed, with_do=True))
        qq, qs, kq, ks, vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize_qkv(q, k, v, layout)
        o, lse = ops.mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, layout, w.scale)
        ref = ops.bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o, lse, do, layout, w.scale)
        got = ops.bf16_attn_bwd_static(qq, qs, kq, ks, vtn, vtn_sc, o, lse, do, layout, w.scale)
        torch.cuda.synchronize()
        for r, g, name in zip(ref, got, ("dq", "dk", "dv")):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16)), (seed, name)
        outs.append(got[0].clone())
    assert not torch.equal(outs[0], outs[1])   # the second call computed its own result
