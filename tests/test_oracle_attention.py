"""Pins for the oracle's causal attention (CPU only).

The oracle is checked against: torch's scaled_dot_product_attention in fp64 (a library routine)
when quantisation is off and both V copies are the same tensor; a pure-Python per-row loop on
tiny inputs with distinct V copies; its own two-partial form (completed block, own block,
log-sum-exp merge); closed forms; the GQA head map; and the causality invariant.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import mx


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _sdpa_ref(q, k, v, scale):
    """torch SDPA, fp64, causal; inputs [B,S,H,D] with equal head counts."""
    qt, kt, vt = (torch.tensor(a).permute(0, 2, 1, 3) for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("S", [1, 31, 32, 33, 100, 160])
def test_no_quantisation_equals_textbook_sdpa(S):
    q, k, v = _rand((2, S, 3, 128), 0), _rand((2, S, 3, 128), 1), _rand((2, S, 3, 128), 2)
    O, L = A.causal_attention(q, k, v, v, 0.088, chunk=64)
    np.testing.assert_allclose(O, _sdpa_ref(q, k, v, 0.088), rtol=0, atol=1e-12)
    s = 0.088 * np.einsum("bihd,bjhd->bhij", q, k)
    s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    lse = torch.logsumexp(torch.tensor(s), dim=-1).numpy()
    np.testing.assert_allclose(L, lse, rtol=0, atol=1e-12)


def _loop_reference(q, k, vc, vt, scale):
    """Pure-Python per-row loop: W_j(i) = vc[j] for j < 32*floor(i/32), else vt[j]."""
    B, S, Hq, D = q.shape
    g = Hq // k.shape[2]
    O = np.zeros_like(q)
    L = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            for i in range(S):
                sc = [scale * sum(q[b, i, h, d] * k[b, j, hk, d] for d in range(D)) for j in range(i + 1)]
                mx_ = max(sc)
                w = [math.exp(x - mx_) for x in sc]
                tot = sum(w)
                L[b, h, i] = mx_ + math.log(tot)
                first_own = 32 * (i // 32)
                for j in range(i + 1):
                    src = vc if j < first_own else vt
                    O[b, i, h, :] += (w[j] / tot) * src[b, j, hk, :]
    return O, L


def test_split_rule_against_loop():
    S, D = 70, 8
    q, k = _rand((1, S, 2, D), 3), _rand((1, S, 1, D), 4)
    vc, vt = _rand((1, S, 1, D), 5), _rand((1, S, 1, D), 6) + 10.0   # far apart: a wrong pick shows
    O, L = A.causal_attention(q, k, vc, vt, 0.3, chunk=16)
    Or, Lr = _loop_reference(q, k, vc, vt, 0.3)
    np.testing.assert_allclose(O, Or, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lr, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S,Hq,Hkv", [(128, 2, 2), (200, 4, 1), (96, 6, 3)])
def test_two_partial_form_equals_direct(S, Hq, Hkv):
    q, k = _rand((1, S, Hq, 128), 7), _rand((1, S, Hkv, 128), 8)
    vc, vt = _rand((1, S, Hkv, 128), 9), _rand((1, S, Hkv, 128), 10)
    O1, L1 = A.causal_attention(q, k, vc, vt, 1 / math.sqrt(128), chunk=64)
    O2, L2 = A.causal_attention_two_partials(q, k, vc, vt, 1 / math.sqrt(128), chunk=48)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-12)


def test_first_block_has_empty_completed_partial():
    # rows < 32 see only their own block: O = textbook attention on the token-normalised copy
    S = 32
    q, k = _rand((1, S, 2, 128), 11), _rand((1, S, 2, 128), 12)
    vc, vt = _rand((1, S, 2, 128), 13), _rand((1, S, 2, 128), 14)
    O, _ = A.causal_attention(q, k, vc, vt, 0.1)
    np.testing.assert_allclose(O, _sdpa_ref(q, k, vt, 0.1), rtol=0, atol=1e-12)
    O2, _ = A.causal_attention_two_partials(q, k, vc, vt, 0.1)
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-12)


def test_gqa_map_equals_repeated_heads():
    S, Hq, Hkv = 96, 8, 2
    q = _rand((1, S, Hq, 128), 15)
    k, vc, vt = (_rand((1, S, Hkv, 128), s) for s in (16, 17, 18))
    O, L = A.causal_attention(q, k, vc, vt, 0.09)
    rep = lambda a: np.repeat(a, Hq // Hkv, axis=2)      # q head h -> kv head h // 4
    O2, L2 = A.causal_attention(q, rep(k), rep(vc), rep(vt), 0.09)
    np.testing.assert_allclose(O, O2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, L2, rtol=0, atol=1e-13)


def test_constant_values_closed_form():
    # V rows all equal to u with entries exact in E4M3 under any scale choice (small integers):
    # both decoded copies equal u, so every output row is u.
    S = 160
    u = np.array([((d % 9) - 4) * 1.0 for d in range(128)])
    v = np.broadcast_to(u, (1, S, 1, 128)).copy()
    q, k = _rand((1, S, 1, 128), 19), _rand((1, S, 1, 128), 20)
    O, _ = A.reference_forward(q.round(2), k.round(2), v, 0.088)
    np.testing.assert_allclose(O[0, :, 0, :], np.broadcast_to(u, (S, 128)), rtol=0, atol=1e-12)


def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("i", [0, 31, 32, 45, 63, 64, 100])
def test_causality_invariant_bit_exact(i):
    S, Hq, Hkv = 128, 2, 1
    q, k, v = _bf16(_rand((1, S, Hq, 128), 21)), _bf16(_rand((1, S, Hkv, 128), 22)), \
        _bf16(_rand((1, S, Hkv, 128), 23))
    O0, L0 = A.reference_forward(q, k, v, 0.088)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, i + 1:] += _bf16(_rand(q2[:, i + 1:].shape, 24))
    k2[:, i + 1:] *= -3.0
    v2[:, i + 1:] += 5.0
    # raise the V amax of i's own block (a later token in that block) and of later blocks
    last_in_block = 32 * (i // 32) + 31
    if last_in_block > i:
        v2[:, last_in_block] *= 1000.0
    v2[:, min(S - 1, last_in_block + 1):] *= 64.0
    O1, L1 = A.reference_forward(q2, k2, v2, 0.088)
    np.testing.assert_array_equal(O1[:, : i + 1], O0[:, : i + 1])
    np.testing.assert_array_equal(L1[:, :, : i + 1], L0[:, :, : i + 1])
    # and the columnwise decode of i's own block really did change (the leak the split avoids)
    if last_in_block > i:
        ct0, cs0 = mx.quantize_colwise(v)
        ct1, cs1 = mx.quantize_colwise(v2)
        assert np.any(cs0[..., i // 32] != cs1[..., i // 32])


def test_leaky_variant_would_change():
    # Negative control on the oracle itself: attending the own block with the columnwise copy
    # makes row i depend on a later token of its block.
    S, i = 64, 40
    q, k, v = _bf16(_rand((1, S, 1, 128), 25)), _bf16(_rand((1, S, 1, 128), 26)), \
        _bf16(_rand((1, S, 1, 128), 27))
    v2 = v.copy(); v2[:, 63] *= 1000.0

    def leaky(vv):
        qc, qs = mx.quantize_rowwise(q); kc, ks = mx.quantize_rowwise(k)
        ct, cs = mx.quantize_colwise(vv)
        vc = mx.dequantize_colwise(ct, cs)
        return A.causal_attention(mx.dequantize_rowwise(qc, qs), mx.dequantize_rowwise(kc, ks),
                                  vc, vc, 0.088)[0]
    assert np.any(leaky(v)[:, i] != leaky(v2)[:, i])


def test_sampled_rows_match_full():
    S = 300
    q, k, vc, vt = (_rand((1, S, 2, 128), s) for s in (28, 29, 30, 31))
    O, L = A.causal_attention(q, k, vc, vt, 0.088, chunk=64)
    rows = np.array([0, 5, 31, 32, 33, 64, 127, 128, 255, 299])
    Os, Ls = A.causal_attention(q, k, vc, vt, 0.088, rows=rows, chunk=4)
    np.testing.assert_allclose(Os, O[:, rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(Ls, L[:, :, rows], rtol=0, atol=1e-13)
