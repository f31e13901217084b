"""Host-side logic that needs no GPU: the binding's argument checks (they raise before any call
into the library) and bench.py's rule for reporting the attention kernel's DRAM traffic (only
while the kernel source matches the one the committed ncu summary was captured on)."""
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
