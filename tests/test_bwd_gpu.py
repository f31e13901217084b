"""GPU backward on decoded operands against the fp64 oracle backward, through the C ABI.

Both sides get the same inputs: the decoded Q, K and token-normalised V (the quantisers are
bit-exact), O and LSE of the oracle's forward rounded to the BF16 and fp32 the call takes, and dO.  The GPU
rounds P and dS to BF16 for its MMAs (relative 2^-9) and accumulates in fp32; its outputs are BF16.
So each element must lie within
    dV: 2^-7 * sum_i P_ij |dO_i|            + half a BF16 ulp
    dK: 2^-7 * scale * sum_i |dS_ij| |Qh_i| + half a BF16 ulp
    dQ: 2^-7 * scale * sum_j |dS_ij| |Kh_j| + half a BF16 ulp
of the oracle (twice the two roundings' bound, summed with absolute values), where |dS| also carries
the fp32 accumulation of dP = dO V^T and of Dlt = <dO, O> (each a sum of D = 128 products: at most
128 * 2^-24 = 2^-17 of its absolute sum), which a cancelling dP - Dlt does not shrink:
    |dS|_ij -> |dS_ij| + 2^-10 P_ij (|dO_i|.|V_j| + |dO_i|.|O_i|)     (2^-10 = 2^-17 / 2^-7).
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
            acc = np.abs(do[b, :, hq]) @ np.abs(vt[b, :, hk]).T + np.sum(np.abs(do[b, :, hq] * o[b, :, hq]), axis=1)[:, None]
            ds = np.abs(p * (dp - np.sum(do[b, :, hq] * o[b, :, hq], axis=1)[:, None])) + 2.0 ** -10 * p * acc
            tv[b, :, hk] += p.T @ np.abs(do[b, :, hq])
            tk[b, :, hk] += scale * ds.T @ np.abs(qh[b, :, hq])
            tq[b, :, hq] += scale * ds @ np.abs(kh[b, :, hk])
    return tq, tk, tv


def _run_and_check(ops, w, seed):
    q, k, v, do = I.make_qkv(w, seed_offset=seed, with_do=True)
    qb, kb, vb, dob = (bshd_np(t, w.layout).astype(np.float64) for t in (q, k, v, do))
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb))
    vc = mx.dequantize_colwise(*mx.quantize_colwise(vb))
    vt = mx.dequantize_token_norm(*mx.quantize_token_norm(vb))
    # the backward's O and LSE inputs: the oracle forward's, rounded to the BF16 / fp32 the call
    # takes, given to both sides
    O, Lo = A.causal_attention(qh, kh, vc, vt, w.scale)
    o_in = I.to_layout(torch.from_numpy(O).to(torch.bfloat16), w.layout)
    l_in = torch.from_numpy(Lo).to(torch.float32)
    og = bshd_np(o_in, w.layout).astype(np.float64)
    lg = l_in.numpy().astype(np.float64)
    qq, qs, kq, ks, _, _, vtn, vtn_sc = ops.mxfp8_quantize_qkv(q.cuda(), k.cuda(), v.cuda(), w.layout)
    dq, dk, dv = ops.bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o_in.cuda(), l_in.cuda(), do.cuda(), w.layout,
                                   w.scale)
    torch.cuda.synchronize()
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


# S = 32 and 96: a single partial tile (every pair is the diagonal one); 160 and 288: a partial last
# tile behind whole ones; 16/4-style grouping with 8/2
@pytest.mark.parametrize("S,Hq,Hkv,layout,B", [(128, 2, 2, I.BSHD, 1), (256, 4, 2, I.BSHD, 1),
                                              (384, 2, 2, I.SBHD, 2), (160, 4, 2, I.BSHD, 1),
                                              (512, 4, 1, I.BSHD, 1), (32, 2, 1, I.BSHD, 1),
                                              (96, 4, 4, I.SBHD, 2), (288, 8, 2, I.BSHD, 1)])
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


def _abs_terms_sampled(qh, kh, vt, o, lse, do, scale, rows, keys):
    """The tolerance terms of _abs_terms (with the same accumulation term in |dS|) at the sampled dQ rows
    and dK, dV keys."""
    B, S, Hq, D = qh.shape
    g = Hq // kh.shape[2]
    tq = np.zeros((B, len(rows), Hq, D))
    tk = np.zeros((B, len(keys), kh.shape[2], D))
    tv = np.zeros_like(tk)
    for b in range(B):
        for hq in range(Hq):
            hk = hq // g
            for n, i in enumerate(rows):
                p = np.exp(scale * (kh[b, : i + 1, hk] @ qh[b, i, hq]) - lse[b, hq, i])
                acc = np.abs(vt[b, : i + 1, hk]) @ np.abs(do[b, i, hq]) + np.sum(np.abs(do[b, i, hq] * o[b, i, hq]))
                ds = np.abs(p * (vt[b, : i + 1, hk] @ do[b, i, hq] - np.dot(do[b, i, hq], o[b, i, hq]))) + 2.0 ** -10 * p * acc
                tq[b, n, hq] = scale * ds @ np.abs(kh[b, : i + 1, hk])
            ri = np.arange(int(keys.min()), S)
            vis = keys[None, :] <= ri[:, None]
            p = np.where(vis, np.exp(np.where(vis, scale * qh[b, ri, hq] @ kh[b, keys, hk].T, 0.0)
                                     - lse[b, hq, ri][:, None]), 0.0)
            acc = np.abs(do[b, ri, hq]) @ np.abs(vt[b, keys, hk]).T + np.sum(np.abs(do[b, ri, hq] * o[b, ri, hq]), axis=1)[:, None]
            ds = np.abs(p * (do[b, ri, hq] @ vt[b, keys, hk].T - np.sum(do[b, ri, hq] * o[b, ri, hq], axis=1)[:, None])) \
                + 2.0 ** -10 * p * acc
            tv[b, :, hk] += p.T @ np.abs(do[b, ri, hq])
            tk[b, :, hk] += scale * ds.T @ np.abs(qh[b, ri, hq])
    return tq, tk, tv


def test_bwd_b2_s32k_sbhd_sampled(ops):
    """B=2, Hq=Hkv=16, S=32768, SBHD (the shape the pages time forward + backward on): dQ at sampled
    rows and dK, dV at sampled keys among the last 512 tokens, query heads 0 and 15, against the
    oracle's sampled backward.  O and LSE of every row those outputs read (the sampled rows and all
    rows from the first sampled key on) come from the oracle's forward, rounded to the BF16 and fp32
    the call takes, and both sides get them; the other rows keep the library forward's values,
    which no checked output reads."""
    w = I.WORKLOADS["mha_b2_s32k_h16_sbhd"]
    S, L = w.S, w.layout
    q, k, v, do = I.make_qkv(w, with_do=True)
    heads = [0, 15]
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 31, 32, 4095, 4096, S - 600, S - 1], rng.integers(0, S, 6)]))
    keys = np.unique(np.concatenate([[S - 512, S - 481, S - 480, S - 129, S - 128, S - 33, S - 32, S - 1],
                                     rng.integers(S - 512, S, 4)]))
    need = np.union1d(rows, np.arange(int(keys.min()), S))
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    qq, qs, kq, ks, vt, vsc, vtn, vtn_sc = ops.mxfp8_quantize_qkv(qd, kd, vd, L)
    o, lse = ops.mxfp8_causal_attn_fwd(qq, qs, kq, ks, vt, vsc, vtn, vtn_sc, L, w.scale, p_terms=2)
    # the oracle's operands for the two heads (quantisation is per row / token / head, so the
    # head slice quantises exactly as the whole tensor does)
    f64 = lambda t: bshd_np(t[:, :, heads], L).astype(np.float64)
    qb, kb, vb, dob = f64(q), f64(k), f64(v), f64(do)
    qh = mx.dequantize_rowwise(*mx.quantize_rowwise(qb))
    kh = mx.dequantize_rowwise(*mx.quantize_rowwise(kb))
    vc = mx.dequantize_colwise(*mx.quantize_colwise(vb))
    vtt = mx.dequantize_token_norm(*mx.quantize_token_norm(vb))
    O_n, L_n = A.causal_attention(qh, kh, vc, vtt, w.scale, rows=need)           # [B,n,2,D], [B,2,n]
    O_bf = torch.from_numpy(O_n).to(torch.bfloat16)
    L_f32 = torch.from_numpy(L_n).to(torch.float32)
    ob = I.to_bshd(o, L)
    nt = torch.from_numpy(need).cuda()
    for j, h in enumerate(heads):
        ob[:, nt, h] = O_bf[:, :, j].cuda()
        lse[:, h, nt] = L_f32[:, j].cuda()
    dq, dk, dv = ops.bf16_attn_bwd(qq, qs, kq, ks, vtn, vtn_sc, o, lse, dod, L, w.scale)
    torch.cuda.synchronize()
    O_full = np.zeros(qh.shape)
    O_full[:, need] = O_bf.float().numpy().astype(np.float64)
    L_full = np.zeros((w.B, len(heads), S))
    L_full[:, :, need] = L_f32.numpy().astype(np.float64)
    rq, rk, rv = A.causal_attention_bwd_sampled(qh, kh, vtt, O_full, L_full, dob, w.scale, rows, keys)
    tq, tk, tv = _abs_terms_sampled(qh, kh, vtt, O_full, L_full, dob, w.scale, rows, keys)
    out = []
    for name, g, sel, r, t in (("dq", dq, rows, rq, tq), ("dk", dk, keys, rk, tk), ("dv", dv, keys, rv, tv)):
        gg = I.to_bshd(g, L)[:, torch.from_numpy(sel).cuda()][:, :, heads].float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(gg)), name
        err = np.abs(gg - r)
        bound = 2.0 ** -7 * t + bf16_half_ulp(r) + 1e-6
        assert np.all(err <= bound), "%s: worst excess %.3e (max err %.3e)" % (name, (err - bound).max(), err.max())
        out.append("%s max %.2e" % (name, err.max()))
    print(", ".join(out))
