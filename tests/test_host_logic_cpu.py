"""Host-side logic that needs no GPU: the binding's argument checks (they raise before any call
into the library), bench.py's rule for reporting the attention kernel's DRAM traffic (only
while the kernel source matches the one the committed ncu summary was captured on), and the
bench's tolerance check on sampled rows and its compulsory-bytes estimate."""
import hashlib
import os

import pytest
import torch

import bench


@pytest.fixture(scope="module")
def ops():
    from block_scaled_causal_gb300 import _binding
    return _binding


def test_binding_rejects_cpu_tensors(ops):
    x = torch.zeros((1, 128, 2, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ops.mxfp8_quantize_qk_rowwise(x)
    with pytest.raises(ValueError):
        ops.mxfp8_quantize_qkv(x, x, x)
    with pytest.raises(ValueError):
        ops.mxfp8_quantize(ops.QUANT_ROWWISE, x)


def test_binding_rejects_wrong_dtype_and_rank(ops):
    with pytest.raises(ValueError):
        ops.mxfp8_quantize_v_colwise(torch.zeros((1, 128, 2, 128), dtype=torch.float32))
    with pytest.raises(ValueError):
        ops._bshd_dims(torch.zeros((128, 2, 128)), ops.BSHD)


def test_layout_dims(ops):
    x = torch.zeros((3, 5, 7, 128))
    assert ops._bshd_dims(x, ops.BSHD) == (3, 5, 7, 128)
    assert ops._bshd_dims(x, ops.SBHD) == (5, 3, 7, 128)


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    root = tmp_path
    (root / "profiles").mkdir()
    src_dir = root / "block_scaled_causal_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    src = src_dir / "attn_fwd.cu"
    src.write_bytes(b"// kernel source\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()
    summary = root / "profiles" / "attn_fwd_gqa_s32k_h16_kv4.md"
    summary.write_text("traffic_bytes_per_launch: 1234567\nattn_fwd_cu_sha256: %s\n" % h)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.recorded_traffic() == 1234567.0
    src.write_bytes(b"// kernel source, edited\n")
    assert bench.recorded_traffic() is None
    os.remove(summary)
    assert bench.recorded_traffic() is None


def _fake_outputs(w, O_rows, L_rows, hq, rows, layout_fn):
    """Full-size O [layout] and LSE [B,Hq,S] tensors holding O_rows / L_rows at (hq, rows)."""
    import numpy as np
    o = torch.zeros((w.B, w.S, w.Hq, w.D), dtype=torch.float32)
    o[:, rows, hq] = torch.from_numpy(O_rows).float()
    lse = torch.zeros((w.B, w.Hq, w.S), dtype=torch.float32)
    lse[:, hq, rows] = torch.from_numpy(L_rows).float()
    return layout_fn(o.to(torch.bfloat16), w.layout), lse


def test_error_rows_applies_the_tolerances():
    """bench.error_rows: max-abs 3e-2 plus half a BF16 ulp of the oracle value, mean-abs 3e-3,
    LSE 1e-3 relative; rows and head are read in the output's own layout."""
    import numpy as np
    from block_scaled_causal_gb300 import inputs as I
    for layout in (I.BSHD, I.SBHD):
        w = I.Workload("t", 2, 64, 3, 1, layout=layout)
        rows = np.array([0, 5, 63])
        hq = 2
        rng = np.random.default_rng(0)
        O = np.round(rng.standard_normal((w.B, len(rows), w.D)) * 64) / 64     # exact in BF16
        L = rng.standard_normal((w.B, len(rows))) + 5.0
        L32 = L.astype(np.float32).astype(np.float64)
        o, lse = _fake_outputs(w, O, L32, hq, rows, I.to_layout)
        e = bench.error_rows(w, o, lse, (O, L32), hq, rows)
        assert e["max_abs"] == 0.0 and e["within"]
        # one element off by 0.05 (> 3e-2 + half ulp for |O| < 8): max-abs fails, mean-abs still fine
        O2 = O.copy()
        O2[0, 1, 7] += 0.05
        o2, _ = _fake_outputs(w, O2, L32, hq, rows, I.to_layout)
        e = bench.error_rows(w, o2, lse, (O, L32), hq, rows)
        assert not e["within"] and abs(e["max_abs"] - 0.05) < 1e-2
        # every element off by 4e-3: mean-abs fails, max-abs passes
        o3, _ = _fake_outputs(w, O + 4.0e-3, L32, hq, rows, I.to_layout)
        e = bench.error_rows(w, o3, lse, (O, L32), hq, rows)
        assert e["max_abs"] < 3e-2 and e["mean_abs"] > 3e-3 and not e["within"]
        # LSE off by 2e-3 relative
        e = bench.error_rows(w, o, lse * (1 + 2e-3), (O, L32), hq, rows)
        assert not e["within"] and e["lse_rel"] > 1e-3


def test_compulsory_bytes():
    from block_scaled_causal_gb300 import inputs as I
    w = I.WORKLOADS["gqa_s32k_h16_kv4"]
    q = 32768 * 16 * 128
    kv = 32768 * 4 * 128
    expect = q * 33 / 32 + 3 * kv * 33 / 32 + 32768 * 16 * (256 + 4)
    assert bench.compulsory_bytes(w) == pytest.approx(expect)
