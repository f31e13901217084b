"""GPU backward on decoded operands against the fp64 oracle backward, through the C ABI.

Both sides get the same inputs: the decoded Q, K and token-normalised V (the quantisers are
bit-exact), the forward's BF16 O and fp32 LSE as the GPU forward returned them, and dO.  The GPU
rounds P and dS to BF16 for its MMAs (relative 2^-9) and accumulates in fp32; its outputs are BF16.
So each element must lie within
    dV: 2^-7 * sum_i P_ij |dO_i|            + half a BF16 ulp
    dK: 2^-7 * scale * sum_i |dS_ij| |Qh_i| + half a BF16 ulp
    dQ: 2^-7 * scale * sum_j |dS_ij| |Kh_j| + half a BF16 ulp
of the oracle (twice the two roundings' bound, summed with absolute values).
"""
import numpy as np
import pytest
import torch

from block_scaled_causal_gb300 import inputs as I
from oracle import attention as A
from oracle import mx
from tests._helpers import bshd_np
from tests.test_attn_gpu import bf16_half_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def _abs_terms(qh, kh, vt, o, lse, do, scale):
    """sum_i P|dO| per (key, d), and sum |dS||Qh|, sum |dS||Kh| (fp64), for the tolerances."""
    B, S, Hq, D = qh.shape
    Hkv = kh.shape[2]
    g = Hq // Hkv
    tv, tk, tq = np.zeros_like(kh), np.zeros_like(kh), np.zeros_like(qh)
    mask = np.tril(np.ones((S, S), dtype=bool))
    for b in range(B):
        for hq in range(Hq):
            hk = hq // g
            s = scale * qh[b, :, hq] @ kh[b, :, hk].T
            p = np.where(mask, np.exp(np.where(mask, s, 0.0) - lse[b, hq][:, None]), 0.0)
            dp = do[b, :, hq] @ vt[b, :, hk].T
            ds = np.abs(p * (dp - np.sum(do[b, :, hq] * o[b, :, hq], axis=1)[:, None]))
            tv[b, :, hk] += p.T @ np.abs(do[b, :, hq])
            tk[b, :, hk] += scale * ds.T @ np.abs(qh[b, :, hq])
            tq[b, :, hq] += scale * ds @ np.abs(kh[b, :, hk])
    return tq, tk, tv


def _run_and_check(ops, w, seed):
    q, k, v, do = I.make_qkv(w, seed_offset=seed, with_do=True)
    o, lse, dq, dk, dv = ops.forward_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), w.layout, w.scale)
    torch.cuda.synchronize()
    qb, kb, vb, dob = (bshd_np(t, w.layout).astype(np.float64) for t in (q, k, v, do))
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb))
    vt = mx.dequantize_token_norm(*mx.quantize_token_norm(vb))
    og = bshd_np(o, w.layout).astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    rq, rk, rv = A.causal_attention_bwd(qh, kh, vt, og, lg, dob, w.scale)
    tq, tk, tv = _abs_terms(qh, kh, vt, og, lg, dob, w.scale)
    out = []
    for name, g, r, t in (("dq", dq, rq, tq), ("dk", dk, rk, tk), ("dv", dv, rv, tv)):
        gg = bshd_np(g, w.layout).astype(np.float64)
        assert np.all(np.isfinite(gg)), name
        err = np.abs(gg - r)
        bound = 2.0 ** -7 * t + bf16_half_ulp(r) + 1e-6
        assert np.all(err <= bound), "%s: worst excess %.3e (max err %.3e)" % (name, (err - bound).max(), err.max())
        out.append("%s max %.2e rel %.2e" % (name, err.max(), err.max() / max(np.abs(r).max(), 1e-30)))
    return ", ".join(out)


@pytest.mark.parametrize("S,Hq,Hkv,layout,B", [(128, 2, 2, I.BSHD, 1), (256, 4, 2, I.BSHD, 1),
                                              (384, 2, 2, I.SBHD, 2), (160, 4, 2, I.BSHD, 1),
                                              (512, 4, 1, I.BSHD, 1)])
def test_bwd_against_oracle(ops, S, Hq, Hkv, layout, B):
    w = I.Workload("bwd", B, S, Hq, Hkv, layout=layout)
    print(_run_and_check(ops, w, 80))


def test_bwd_heavy_v(ops):
    w = I.Workload("bwd", 1, 256, 2, 2, v_pattern="every7x16")
    print(_run_and_check(ops, w, 81))


def test_bwd_dq_causal_bit_exact(ops):
    """dQ of rows <= i does not change when tokens after i change (their q, k, v and dO)."""
    w = I.Workload("c", 1, 384, 4, 2)
    q, k, v, do = I.make_qkv(w, seed_offset=82, with_do=True)
    base = ops.forward_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), w.layout, w.scale)
    for i in (31, 32, 100, 127, 200):
        q2, k2, v2, do2 = q.clone(), k.clone(), v.clone(), do.clone()
        q2[:, i + 1:] = -q2[:, i + 1:]
        k2[:, i + 1:] = 2.0 * k2[:, i + 1:]
        v2[:, i + 1:] = v2[:, i + 1:] * 16.0
        do2[:, i + 1:] = 0.5 * do2[:, i + 1:]
        pert = ops.forward_backward(q2.cuda(), k2.cuda(), v2.cuda(), do2.cuda(), w.layout, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(base[2][:, : i + 1].view(torch.int16), pert[2][:, : i + 1].view(torch.int16)), i
