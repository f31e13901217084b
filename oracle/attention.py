"""Test infrastructure only: plain CPU fp64 oracle for leak-free causal MXFP8 attention forward.

Nothing in the product path may import this module; only the tests, the smoke check and the
CPU-baseline leg of the benchmark use it.

What it follows ("[PyTorch] Add causal MXFP8 attention without future-token leakage through V
scales", TransformerEngine PR #3865, Description, and the PR's own commit message):

* Q and K enter decoded from their rowwise MXFP8 bytes: Qh, Kh.
* For query token i, blk(i) = 32 * floor(i / 32) is the first token of its own 32-token block.
* Keys j < blk(i) ("completed blocks") are attended with V decoded from its columnwise MXFP8
  quantisation, Vc; every V scale involved covers tokens < blk(i) only.
* Keys blk(i) <= j <= i (the query's own block, at most 32 keys) are attended with V decoded from
  the token-normalised copy, Vt.
* The two partial results are merged through their log-sum-exps.

With s_ij = scale * <Qh_i, Kh_j> this gives, for each row,
    LSE_i = ln sum_{j<=i} exp(s_ij),
    O_i   = sum_{j<=i} exp(s_ij - LSE_i) * W_j(i),  W_j(i) = Vc_j if j < blk(i) else Vt_j,
which `causal_attention` computes directly (the "plain definition"), and
`causal_attention_two_partials` computes in the pages' order: the completed-block partial
(O_c, LSE_c), the own-block partial (O_o, LSE_o), then the log-sum-exp merge.  The two must agree
to fp64 round-off.

GQA: query head hq reads key/value head hq // (Hq / Hkv) (contiguous groups).
P (the softmax weights) is not quantised here: the oracle is the exact result on the decoded
operands.  All arithmetic is fp64; matrix products use numpy's matmul as a library primitive.
Arrays are [B, S, H, D] (canonical order); LSE is [B, Hq, S] in natural log.
"""
from __future__ import annotations

import numpy as np

OWN_BLOCK = 32


def _rows_iter(S: int, rows, chunk: int):
    if rows is None:
        for r0 in range(0, S, chunk):
            yield np.arange(r0, min(S, r0 + chunk))
    else:
        rows = np.asarray(rows, dtype=np.int64)
        for c0 in range(0, len(rows), chunk):
            yield rows[c0:c0 + chunk]


def causal_attention(qh, kh, vc, vt, scale, rows=None, chunk=256):
    """Direct form.  qh [B,S,Hq,D]; kh, vc, vt [B,S,Hkv,D] (decoded, fp64).

    rows: optional 1-D array of query rows to evaluate (default: all S rows).
    Returns O [B,len(rows),Hq,D] and LSE [B,Hq,len(rows)].
    """
    qh, kh, vc, vt = (np.asarray(a, dtype=np.float64) for a in (qh, kh, vc, vt))
    B, S, Hq, D = qh.shape
    Hkv = kh.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    nrows = S if rows is None else len(rows)
    O = np.zeros((B, nrows, Hq, D))
    LSE = np.zeros((B, Hq, nrows))
    for b in range(B):
        for hq in range(Hq):
            hk = hq // g
            out0 = 0
            for ri in _rows_iter(S, rows, chunk):
                kmax = int(ri.max()) + 1
                s = scale * (qh[b, ri, hq, :] @ kh[b, :kmax, hk, :].T)        # [R, kmax]
                i = ri[:, None]
                j = np.arange(kmax)[None, :]
                visible = j <= i
                s = np.where(visible, s, -np.inf)
                m = np.max(s, axis=1, keepdims=True)
                lse = m[:, 0] + np.log(np.sum(np.exp(s - m), axis=1))
                p = np.exp(s - lse[:, None])                                  # 0 where masked
                completed = j < (i // OWN_BLOCK) * OWN_BLOCK
                own = visible & ~completed
                o = np.where(completed, p, 0.0) @ vc[b, :kmax, hk, :] \
                    + np.where(own, p, 0.0) @ vt[b, :kmax, hk, :]
                n = len(ri)
                O[b, out0:out0 + n, hq, :] = o
                LSE[b, hq, out0:out0 + n] = lse
                out0 += n
    return O, LSE


def _partial(s, mask, v):
    """Softmax partial over the keys in mask: (O_part, LSE_part); empty -> (0, -inf)."""
    s = np.where(mask, s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    lsum = np.sum(e, axis=1)
    lse = np.where(empty, -np.inf, m_safe[:, 0] + np.log(np.where(empty, 1.0, lsum)))
    o = (e @ v) / np.where(empty, 1.0, lsum)[:, None]
    return o, lse


def causal_attention_two_partials(qh, kh, vc, vt, scale, rows=None, chunk=256):
    """Two-partial form: completed-block partial, own-block partial, log-sum-exp merge."""
    qh, kh, vc, vt = (np.asarray(a, dtype=np.float64) for a in (qh, kh, vc, vt))
    B, S, Hq, D = qh.shape
    Hkv = kh.shape[2]
    g = Hq // Hkv
    nrows = S if rows is None else len(rows)
    O = np.zeros((B, nrows, Hq, D))
    LSE = np.zeros((B, Hq, nrows))
    for b in range(B):
        for hq in range(Hq):
            hk = hq // g
            out0 = 0
            for ri in _rows_iter(S, rows, chunk):
                kmax = int(ri.max()) + 1
                s = scale * (qh[b, ri, hq, :] @ kh[b, :kmax, hk, :].T)
                i = ri[:, None]
                j = np.arange(kmax)[None, :]
                blk = (i // OWN_BLOCK) * OWN_BLOCK
                o_c, lse_c = _partial(s, j < blk, vc[b, :kmax, hk, :])
                o_o, lse_o = _partial(s, (j >= blk) & (j <= i), vt[b, :kmax, hk, :])
                lse = np.logaddexp(lse_c, lse_o)
                w_c = np.exp(lse_c - lse)                 # exp(-inf) = 0 for an empty partial
                w_o = np.exp(lse_o - lse)
                o = w_c[:, None] * o_c + w_o[:, None] * o_o
                n = len(ri)
                O[b, out0:out0 + n, hq, :] = o
                LSE[b, hq, out0:out0 + n] = lse
                out0 += n
    return O, LSE


def reference_forward(q, k, v, scale, rows=None, chunk=256):
    """Quantise bf16-valued inputs with the oracle's own quantisers, decode, and attend.

    q [B,S,Hq,D], k, v [B,S,Hkv,D] given as fp32/fp64 arrays holding bf16 values.
    Returns (O, LSE) of `causal_attention`.
    """
    from . import mx
    qc, qs = mx.quantize_rowwise(q)
    kc, ks = mx.quantize_rowwise(k)
    vcc, vcs = mx.quantize_colwise(v)
    vtc, vts = mx.quantize_token_norm(v)
    return causal_attention(mx.dequantize_rowwise(qc, qs), mx.dequantize_rowwise(kc, ks),
                            mx.dequantize_colwise(vcc, vcs), mx.dequantize_token_norm(vtc, vts),
                            scale, rows=rows, chunk=chunk)


def causal_attention_bwd(qh, kh, vt, o, lse, do, scale, chunk=256):
    """Backward of the leak-free causal attention on decoded operands, fp64.

    Follows "[PyTorch] Add causal MXFP8 attention without future-token leakage through V scales"
    (TransformerEngine PR #3865), Description, Backward: an FP16/BF16 attention backward on Q and
    K decoded from their rowwise MXFP8 bytes and V decoded from the token-normalised copy, fed
    with the forward's O and LSE.  With s_ij = scale * <Qh_i, Kh_j> (j <= i):
        P_ij  = exp(s_ij - LSE_i)
        dV_j  = sum_i P_ij dO_i               dP_ij = <dO_i, Vt_j>
        Dlt_i = <dO_i, O_i>                   dS_ij = P_ij (dP_ij - Dlt_i)
        dQ_i  = scale * sum_j dS_ij Kh_j      dK_j  = scale * sum_i dS_ij Qh_i
    GQA: dK and dV of a KV head sum over the query heads that read it.

    qh, do, o [B,S,Hq,D]; kh, vt [B,S,Hkv,D]; lse [B,Hq,S].  Returns dq [B,S,Hq,D] and
    dk, dv [B,S,Hkv,D].
    """
    qh, kh, vt, o, lse, do = (np.asarray(a, dtype=np.float64) for a in (qh, kh, vt, o, lse, do))
    B, S, Hq, D = qh.shape
    Hkv = kh.shape[2]
    g = Hq // Hkv
    dq = np.zeros_like(qh)
    dk = np.zeros_like(kh)
    dv = np.zeros_like(vt)
    for b in range(B):
        for hq in range(Hq):
            hk = hq // g
            dlt = np.sum(do[b, :, hq, :] * o[b, :, hq, :], axis=1)            # [S]
            for r0 in range(0, S, chunk):
                ri = np.arange(r0, min(S, r0 + chunk))
                kmax = int(ri.max()) + 1
                s = scale * (qh[b, ri, hq, :] @ kh[b, :kmax, hk, :].T)         # [R, kmax]
                visible = np.arange(kmax)[None, :] <= ri[:, None]
                p = np.where(visible, np.exp(np.where(visible, s, 0.0) - lse[b, hq, ri][:, None]), 0.0)
                dv[b, :kmax, hk, :] += p.T @ do[b, ri, hq, :]
                dp = do[b, ri, hq, :] @ vt[b, :kmax, hk, :].T
                ds = p * (dp - dlt[ri][:, None])
                dq[b, ri, hq, :] += scale * (ds @ kh[b, :kmax, hk, :])
                dk[b, :kmax, hk, :] += scale * (ds.T @ qh[b, ri, hq, :])
    return dq, dk, dv


def causal_attention_bwd_sampled(qh, kh, vt, o, lse, do, scale, rows, keys):
    """causal_attention_bwd restricted to dQ at the query `rows` and dK, dV at the key positions
    `keys`, by the same formulas (PR #3865 page, Description, Backward).  dQ_i reads row i's O and
    LSE; dK_j and dV_j sum over every row i >= j and read those rows' O and LSE, so only they need
    to be meaningful in `o` and `lse`.

    qh, do, o [B,S,Hq,D]; kh, vt [B,S,Hkv,D]; lse [B,Hq,S].  Returns dq [B,len(rows),Hq,D] and
    dk, dv [B,len(keys),Hkv,D].
    """
    qh, kh, vt, o, lse, do = (np.asarray(a, dtype=np.float64) for a in (qh, kh, vt, o, lse, do))
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)
    B, S, Hq, D = qh.shape
    Hkv = kh.shape[2]
    g = Hq // Hkv
    dq = np.zeros((B, len(rows), Hq, D))
    dk = np.zeros((B, len(keys), Hkv, D))
    dv = np.zeros((B, len(keys), Hkv, D))
    for b in range(B):
        for hq in range(Hq):
            hk = hq // g
            for n, i in enumerate(rows):
                s = scale * (kh[b, : i + 1, hk, :] @ qh[b, i, hq, :])                 # keys j <= i
                p = np.exp(s - lse[b, hq, i])
                dp = vt[b, : i + 1, hk, :] @ do[b, i, hq, :]
                ds = p * (dp - np.dot(do[b, i, hq, :], o[b, i, hq, :]))
                dq[b, n, hq, :] = scale * (ds @ kh[b, : i + 1, hk, :])
            if len(keys) == 0:
                continue
            ri = np.arange(int(keys.min()), S)                                      # rows i >= min key
            s = scale * (qh[b, ri, hq, :] @ kh[b, keys, hk, :].T)                   # [R, K]
            visible = keys[None, :] <= ri[:, None]
            p = np.where(visible, np.exp(np.where(visible, s, 0.0) - lse[b, hq, ri][:, None]), 0.0)
            dp = do[b, ri, hq, :] @ vt[b, keys, hk, :].T
            ds = p * (dp - np.sum(do[b, ri, hq, :] * o[b, ri, hq, :], axis=1)[:, None])
            dv[b, :, hk, :] += p.T @ do[b, ri, hq, :]
            dk[b, :, hk, :] += scale * (ds.T @ qh[b, ri, hq, :])
    return dq, dk, dv
