"""The bench's roofline arithmetic on the CPU: the per-layer byte and multiply-add counts behind
every `frac` it prints, pinned to values worked out by hand from the layer's widths, and the
choice of the binding bound."""
import os
import sys
from types import SimpleNamespace

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

H, I = 7168, 2048


def test_expert_bytes_are_codes_plus_scales():
    # gate, up and down each hold I x H E2M1 codes (half a byte) and one E8M0 scale per 32
    assert bench.expert_bytes(H, I) == 3 * (2048 * 7168 // 2) + 3 * (2048 * 7168 // 32) == 23_396_352


def test_decode_layer_bytes_by_hand():
    # 8 experts' weights, x (E4M3 + scales), h twice (E4M3 + scales for 8 pairs), the fp32 expert
    # outputs twice, ids and weights, y in bf16
    weights = 8 * 23_396_352
    x = 7168 + 7168 // 32
    h = 8 * 2048 + 8 * (2048 // 32)
    d = 8 * 7168 * 4
    assert bench.layer_bytes(H, I, 1, 8, 8, True) == weights + x + 2 * h + 2 * d + 8 * 8 + 7168 * 2 == 187_685_152


def test_bf16_layer_bytes_count_two_bytes_and_no_scales():
    weights = 16 * 23_396_352
    x = 2 * 7168 * 2
    h = 16 * 2048 * 2
    assert bench.layer_bytes(H, I, 2, 8, 16, False) == weights + x + 2 * h + 2 * 16 * 7168 * 4 + 16 * 8 + 2 * 7168 * 2


def test_layer_fmas_one_per_weight_per_pair():
    assert bench.layer_fmas(H, I, 1, 8) == 8 * (2048 * 7168 * 2 + 7168 * 2048)
    assert bench.layer_fmas(H, I, 16, 8) == 5_637_144_576


def test_fma_peak():
    assert bench.fma_peak(152, 2070) == pytest.approx(152 * 128 * 2.07e9)


def run(alg_bytes, fmas, chunk=False):
    return SimpleNamespace(alg_bytes=alg_bytes, fmas=fmas, flops=2.0 * fmas, chunk=chunk)


def test_one_row_decode_is_hbm_bound():
    r = bench.bound_of(run(187_685_152, bench.layer_fmas(H, I, 1, 8)), 48.0, 6787.6, 2070.0, 152)
    assert r["bound"] == "hbm"
    assert r["hbm_us"] == pytest.approx(27.65, abs=0.01)
    assert r["frac"] == pytest.approx(187_685_152 / 6787.6e9 / 48e-6, abs=1e-4)
    assert r["alu_us"] == pytest.approx(8.75, abs=0.01)


def test_sixteen_shared_rows_are_fma_bound():
    fmas = bench.layer_fmas(H, I, 16, 8)
    r = bench.bound_of(run(195_400_192, fmas), 328.0, 6787.6, 2070.0, 152)
    assert r["bound"] == "alu"
    assert r["alu_us"] == pytest.approx(fmas / (152 * 128 * 2.07e9) * 1e6, abs=0.01)
    assert r["frac"] == pytest.approx(139.97 / 328.0, abs=1e-3)


def test_chunk_takes_the_longer_of_bytes_and_tensor_flops(monkeypatch):
    monkeypatch.setattr(bench, "tensor_peak_fp8", lambda: (3817.0, "test"))
    fmas = bench.layer_fmas(H, I, 4096, 8)
    r = bench.bound_of(run(8_096_186_368, fmas, chunk=True), 2106.0, 6787.6, 2070.0, 152)
    assert r["tensor_us"] == pytest.approx(2.0 * fmas / 3817e12 * 1e6, abs=0.01)
    assert r["bound"] == "hbm" and r["hbm_us"] > r["tensor_us"]
    r = bench.bound_of(run(1_000_000, fmas, chunk=True), 2106.0, 6787.6, 2070.0, 152)
    assert r["bound"] == "tensor"
