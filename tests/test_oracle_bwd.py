"""Pins of the oracle's attention backward (CPU, fp64).

* With the own block and the completed blocks on the same V (so the forward is plain causal
  softmax attention) and O, LSE from the oracle forward, the backward is the exact gradient of
  L = sum(dO * O) with respect to the decoded Q, K and V: checked against central finite
  differences of the oracle forward, which shares no arithmetic with the backward formulas.
* GQA: dK, dV of a KV head equal the sums of the per-head gradients of the MHA problem with K, V
  repeated over the group.
* Causality: dQ of row i does not change when tokens after i change; dK, dV of token j do not
  change when queries before j change.
"""
import numpy as np
import pytest

from oracle import attention as A

pytestmark = pytest.mark.filterwarnings("ignore")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _loss(q, k, v, do, scale):
    O, _ = A.causal_attention(q, k, v, v, scale)
    return float(np.sum(O * do))


@pytest.mark.parametrize("S,Hq,Hkv,D", [(5, 1, 1, 3), (9, 2, 1, 4), (40, 2, 2, 3)])
def test_bwd_matches_finite_differences(S, Hq, Hkv, D):
    B, scale = 1, 0.7
    q, k, v = _rand((B, S, Hq, D), 1), _rand((B, S, Hkv, D), 2), _rand((B, S, Hkv, D), 3)
    do = _rand((B, S, Hq, D), 4)
    O, L = A.causal_attention(q, k, v, v, scale)
    dq, dk, dv = A.causal_attention_bwd(q, k, v, O, L, do, scale)
    h = 1e-6
    rng = np.random.default_rng(5)
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(q, k, v, do, scale)
            arr[idx] = old - h
            lm = _loss(q, k, v, do, scale)
            arr[idx] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def test_bwd_gqa_is_sum_over_group():
    B, S, Hq, Hkv, D, scale = 1, 33, 4, 2, 5, 0.3
    q, k, v = _rand((B, S, Hq, D), 11), _rand((B, S, Hkv, D), 12), _rand((B, S, Hkv, D), 13)
    do = _rand((B, S, Hq, D), 14)
    O, L = A.causal_attention(q, k, v, v, scale)
    dq, dk, dv = A.causal_attention_bwd(q, k, v, O, L, do, scale)
    kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    dq2, dk2, dv2 = A.causal_attention_bwd(q, kr, vr, O, L, do, scale)
    np.testing.assert_allclose(dq, dq2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk, dk2.reshape(B, S, Hkv, Hq // Hkv, D).sum(axis=3), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(B, S, Hkv, Hq // Hkv, D).sum(axis=3), rtol=1e-12, atol=1e-12)


def test_bwd_causality():
    B, S, H, D, scale, i = 1, 48, 2, 4, 0.5, 20
    q, k, v = _rand((B, S, H, D), 21), _rand((B, S, H, D), 22), _rand((B, S, H, D), 23)
    do = _rand((B, S, H, D), 24)
    O, L = A.causal_attention(q, k, v, v, scale)
    dq, dk, dv = A.causal_attention_bwd(q, k, v, O, L, do, scale)
    # tokens after i change (their q, k, v, dO, O, LSE): dQ of rows <= i is unchanged
    k2, v2 = k.copy(), v.copy()
    k2[:, i + 1:] += 3.0
    v2[:, i + 1:] *= -2.0
    O2, L2 = A.causal_attention(q, k2, v2, v2, scale)
    dq2, _, _ = A.causal_attention_bwd(q, k2, v2, O2, L2, do, scale)
    np.testing.assert_array_equal(dq[:, : i + 1], dq2[:, : i + 1])
    # queries before j = i change: dK, dV of tokens >= i are unchanged
    q3, do3 = q.copy(), do.copy()
    q3[:, :i] += 1.5
    do3[:, :i] *= 0.25
    O3, L3 = A.causal_attention(q3, k, v, v, scale)
    _, dk3, dv3 = A.causal_attention_bwd(q3, k, v, O3, L3, do3, scale)
    np.testing.assert_allclose(dk[:, i:], dk3[:, i:], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dv[:, i:], dv3[:, i:], rtol=1e-13, atol=1e-13)


def test_bwd_sampled_matches_full():
    """The sampled backward gives the full backward's dQ rows and dK, dV keys (GQA, B=2), including
    the first and last rows and keys on both sides of a 32-token block edge."""
    B, S, Hq, Hkv, D, scale = 2, 96, 4, 2, 8, 0.4
    q, k, v = _rand((B, S, Hq, D), 31), _rand((B, S, Hkv, D), 32), _rand((B, S, Hkv, D), 33)
    do = _rand((B, S, Hq, D), 34)
    O, L = A.causal_attention(q, k, v, v, scale)
    dq, dk, dv = A.causal_attention_bwd(q, k, v, O, L, do, scale)
    rows, keys = np.array([0, 5, 31, 32, 50, 95]), np.array([0, 31, 32, 64, 90, 95])
    sq, sk, sv = A.causal_attention_bwd_sampled(q, k, v, O, L, do, scale, rows, keys)
    np.testing.assert_allclose(sq, dq[:, rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sk, dk[:, keys], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sv, dv[:, keys], rtol=1e-12, atol=1e-12)
    # only the rows the sampled outputs read matter: garbage elsewhere changes nothing
    keys2 = np.array([64, 90, 95])
    sq, sk, sv = A.causal_attention_bwd_sampled(q, k, v, O, L, do, scale, rows, keys2)
    O2, L2 = O.copy(), L.copy()
    other = np.setdiff1d(np.arange(S), np.concatenate([rows, np.arange(keys2.min(), S)]))
    assert len(other) > 40
    O2[:, other] = 1e3
    L2[:, :, other] = -7.0
    tq, tk, tv = A.causal_attention_bwd_sampled(q, k, v, O2, L2, do, scale, rows, keys2)
    np.testing.assert_array_equal(tq, sq)
    np.testing.assert_array_equal(tk, sk)
    np.testing.assert_array_equal(tv, sv)
