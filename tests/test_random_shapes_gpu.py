"""A seeded sweep of random small shapes, through the C ABI, against the oracle: the one-launch
quantiser bit for bit (Q, K rowwise; V columnwise and token-normalised), the attention forward
within the tolerance (both P modes, so both softmax forms of the kernel) and, on six of the shapes,
the backward within its bound, the causality invariant bit for bit, the MXFP8 O epilogue and the
leaky control, over batch sizes,
sequence lengths that are any multiple of 32 (partial last tiles, single-block sequences), head
ratios (MHA and GQA up to 8:1) and both layouts.  The shapes are drawn once from a fixed seed, so the
sweep is the same on every run."""
import numpy as np
import pytest
import torch

from block_scaled_causal_gb300 import inputs as I
from tests import test_attn_gpu as T
from tests import test_quant_gpu as Q

pytestmark = pytest.mark.gpu


def _shapes(n=10, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(rng.integers(1, 4))
        S = 32 * int(rng.integers(1, 21))              # 32 .. 640
        Hkv = int(rng.choice([1, 2, 3]))
        g = int(rng.choice([1, 2, 4, 8]))
        layout = int(rng.choice([I.BSHD, I.SBHD]))
        out.append((B, S, Hkv * g, Hkv, layout))
    return out


SHAPES = _shapes()


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


@pytest.mark.parametrize("B,S,Hq,Hkv,layout", SHAPES)
def test_quantiser_bit_exact(ops, B, S, Hq, Hkv, layout):
    w = I.Workload("r", B, S, Hq, Hkv, layout=layout)
    q, k, v = I.make_qkv(w, seed_offset=S + 7 * Hq)
    Q._check_rowwise(ops, q, layout)
    Q._check_rowwise(ops, k, layout)
    Q._check_v(ops, v, layout)
    # the one-launch quantiser writes the same bytes as the dedicated calls
    fused = ops.mxfp8_quantize_qkv(q.cuda(), k.cuda(), v.cuda(), layout)
    separate = (*ops.mxfp8_quantize_qk_rowwise(q.cuda(), layout), *ops.mxfp8_quantize_qk_rowwise(k.cuda(), layout),
                *ops.mxfp8_quantize_v_fused(v.cuda(), layout))
    torch.cuda.synchronize()
    for x, y in zip(fused, separate):
        assert torch.equal(x, y)


@pytest.mark.parametrize("B,S,Hq,Hkv,layout", SHAPES)
@pytest.mark.parametrize("p_terms", [1, 2])
def test_forward_within_tolerance(ops, B, S, Hq, Hkv, layout, p_terms):
    w = I.Workload("r", B, S, Hq, Hkv, layout=layout)
    q, k, v = I.make_qkv(w, seed_offset=S + 7 * Hq)
    Og, Lg = T._run(ops, w, q, k, v, p_terms)
    O, L = T._oracle(w, q, k, v)
    print(T._compare(Og, Lg, O, L))


@pytest.mark.parametrize("B,S,Hq,Hkv,layout", SHAPES[:6])
def test_backward_within_tolerance(ops, B, S, Hq, Hkv, layout):
    # the backward's own per-element bound (tests/test_bwd_gpu.py): BF16 P and dS for the MMAs,
    # fp32 accumulation, BF16 outputs
    from tests import test_bwd_gpu as BW
    w = I.Workload("r", B, S, Hq, Hkv, layout=layout)
    print(BW._run_and_check(ops, w, S + 11 * Hq))


@pytest.mark.parametrize("B,S,Hq,Hkv,layout", SHAPES[:6])
@pytest.mark.parametrize("p_terms", [1, 2])
def test_causality_bit_exact(ops, B, S, Hq, Hkv, layout, p_terms):
    # every token after a random row i perturbed (q, k, v, and the V amax of i's own 32-block
    # raised): rows <= i of O and LSE stay bit-identical, in either layout and P mode
    w = I.Workload("r", B, S, Hq, Hkv, layout=layout)
    q, k, v = I.make_qkv(w, seed_offset=S + 7 * Hq)
    rng = np.random.default_rng(S * 31 + Hq)
    o0, l0 = ops.forward(q.cuda(), k.cuda(), v.cuda(), layout, w.scale, p_terms=p_terms)
    for i in sorted({int(rng.integers(0, S - 1)), S // 2 - 1, 32 * (S // 64)}):
        qb, kb, vb = (I.to_bshd(t, layout) for t in (q, k, v))
        q2, k2, v2 = (I.to_layout(t, layout).contiguous() for t in T._perturb_after(qb, kb, vb, i))
        o1, l1 = ops.forward(q2.cuda(), k2.cuda(), v2.cuda(), layout, w.scale, p_terms=p_terms)
        torch.cuda.synchronize()
        a, b = I.to_bshd(o0, layout)[:, : i + 1], I.to_bshd(o1, layout)[:, : i + 1]
        assert torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16)), i
        assert torch.equal(l0[..., : i + 1].contiguous().view(torch.int32), l1[..., : i + 1].contiguous().view(torch.int32)), i


@pytest.mark.parametrize("B,S,Hq,Hkv,layout", SHAPES[:6])
def test_mxfp8_o_and_leaky_control(ops, B, S, Hq, Hkv, layout):
    # the MXFP8 O epilogue (its value and rule checks, tests/test_o8_gpu.py) and the leaky control
    # (own block on the columnwise V as well) against the leaky oracle
    from oracle import attention as A
    from tests import test_o8_gpu as O8
    w = I.Workload("r", B, S, Hq, Hkv, layout=layout)
    q, k, v = I.make_qkv(w, seed_offset=S + 7 * Hq)
    o, o8, osc = O8._run(ops, w, q, k, v)
    O8._check(w, o, o8, osc, O8._oracle(w, q, k, v)[0])
    Og, Lg = T._run(ops, w, q, k, v, 2, leaky=1)
    qh, kh, vc, _ = T._oracle_operands(w, q, k, v, None)
    O, L = A.causal_attention(qh, kh, vc, vc, w.scale)
    print(T._compare(Og, Lg, O, L))
