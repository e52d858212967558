"""Pins of the oracle's element formats and quantiser against things other than itself:
the OCP MX v1.0 E2M1 value table, torch's float8 / bf16 casts (library routines), and
hand-worked quantiser cases."""
import math

import numpy as np
import pytest
import torch


# OCP Microscaling Formats (MX) v1.0, FP4 E2M1: the eight magnitudes the spec lists.
E2M1_SPEC = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_all_codes_match_spec_table(orc):
    for c in range(16):
        v = orc.e2m1_value(c)
        ref = E2M1_SPEC[c & 7]
        assert abs(v) == ref
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_e4m3_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = orc.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9


def test_ue8m0_scales(orc):
    for c in range(255):
        assert orc.ue8m0_value(c) == 2.0 ** (c - 127)
    assert math.isnan(orc.ue8m0_value(255))
    if hasattr(torch, "float8_e8m0fnu"):
        codes = torch.arange(255, dtype=torch.int32).to(torch.uint8)
        ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert all(orc.ue8m0_value(c) == ref[c] for c in range(255))


def _edge_floats():
    vals = [0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 3.4028234663852886e38, 1e-45, -1e-45, 1.17549435e-38,
            float("inf"), float("-inf")]
    bits = [0x3F808000, 0x3F818000, 0x3F80FFFF, 0x3F817FFF, 0x7F7FFFFF, 0x00008000, 0x00018000, 0x807FFFFF]
    vals += [np.uint32(b).view(np.float32).item() for b in bits]
    return np.array(vals, np.float32)


def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(5)
    a = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    a = a[~np.isnan(a)]
    a = np.concatenate([a, _edge_floats()])
    got = orc.f32_to_bf16(a)
    ref = torch.from_numpy(a.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    nan = orc.f32_to_bf16(np.array([np.nan], np.float32))
    assert (nan[0] & 0x7F80) == 0x7F80 and (nan[0] & 0x7F) != 0


def test_e4m3_encode_matches_torch(orc):
    rng = np.random.default_rng(6)
    ex = rng.integers(-14, 10, size=40000)
    v = (rng.uniform(1, 2, size=ex.size) * np.exp2(ex) * rng.choice([-1, 1], size=ex.size)).astype(np.float32)
    # exact midpoints between neighbouring codes (ties) and the saturation edge
    grid = np.array([orc.e4m3_value(c) for c in range(0x7F)])
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, np.array([447.9, 448.0, 449.0, 463.9, 464.0, 500.0, 1e9, 0.0, -0.0], np.float32)])
    got = orc.e4m3_encode(v.astype(np.float64))
    ref = torch.from_numpy(np.clip(v, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    assert orc.e4m3_encode([np.nan])[0] == 0x7F


def test_quantiser_hand_cases(orc):
    # amax = 56 = 448 * 2^-3: shared exponent floor(log2 56) - 8 = -3 -> scale code 124; 56 maps to 448 exactly.
    h = np.zeros(32, np.float32)
    h[0] = 56.0
    h[1] = -7.0           # -7 / 2^-3 = -56 -> E4M3 -56 exactly (1.75 * 2^5): code 0x80 | (12 << 3) | 6
    codes, sc = orc.quant_e4m3(h)
    assert sc[0] == 124 and codes[0] == 0x7E and codes[1] == (0x80 | (12 << 3) | 6) and codes[2] == 0
    # ties to even under scale 2^0 (amax 256 -> exponent 8 - 8 = 0 -> code 127)
    h = np.zeros(32, np.float32)
    h[0] = 256.0
    h[1] = 1.0625          # halfway 1.0 (mantissa 000) / 1.125 (001) -> 1.0 = 0x38
    h[2] = 1.1875          # halfway 1.125 (001) / 1.25 (010) -> 1.25 = 0x3A
    h[3] = -2.0 ** -10     # halfway 0 / 2^-9 -> -0 = 0x80
    codes, sc = orc.quant_e4m3(h)
    assert sc[0] == 127 and list(codes[:4]) == [0x78, 0x38, 0x3A, 0x80]
    # saturation: amax 480 has exponent 8 -> scale 2^0; 480 > 448 saturates to 0x7E
    h = np.zeros(32, np.float32)
    h[5] = -480.0
    codes, sc = orc.quant_e4m3(h)
    assert sc[0] == 127 and codes[5] == 0xFE
    # all zero (one negative zero): scale code 127, zero codes keep their sign
    h = np.zeros(32, np.float32)
    h[3] = -0.0
    codes, sc = orc.quant_e4m3(h)
    assert sc[0] == 127 and codes[3] == 0x80 and codes[0] == 0
    # NaN or Inf anywhere in the block: NaN scale
    for bad in (np.nan, np.inf, -np.inf):
        h = np.ones(32, np.float32)
        h[7] = bad
        codes, sc = orc.quant_e4m3(h)
        assert sc[0] == 0xFF
    # tiny amax clamps the scale code at 0 (2^-127); elements are still representable
    h = np.zeros(32, np.float32)
    h[0] = np.float32(2.0 ** -130)
    codes, sc = orc.quant_e4m3(h)
    assert sc[0] == 0 and orc.e4m3_value(int(codes[0])) == 2.0 ** -3


def test_quantiser_matches_library_cast_on_gaussian_blocks(orc):
    """The oracle's block quantiser against torch's float8 cast under the same E8M0 choice,
    computed here with numpy's frexp (a different implementation of the same OCP MX rule)."""
    rng = np.random.default_rng(7)
    h = (rng.standard_normal(32 * 512) * np.exp2(rng.integers(-20, 20, size=32 * 512 // 32).repeat(32))).astype(np.float32)
    codes, sc = orc.quant_e4m3(h)
    blocks = h.reshape(-1, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=1)
    _, e2 = np.frexp(amax)
    ref_sc = np.clip(e2 - 1 - 8 + 127, 0, 254)
    assert np.array_equal(sc, ref_sc.astype(np.uint8))
    v = np.clip(blocks / np.exp2(ref_sc - 127)[:, None], -448, 448).astype(np.float32).ravel()
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
