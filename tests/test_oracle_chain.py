"""Pins of the oracle's arithmetic: hand-derived evaluation-order cases (tests/golden),
one-hot layouts, exact integer sums, brute force against torch float64 matmul (a library
routine, with an independent dequantisation written here), the fp32 chain within the
float64 bound, the epilogue's special values, and the combine."""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "chain_order.json")

E2M1_SPEC = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def _bf16_bits(v):
    return int(np.array([v], np.float32).view(np.uint32)[0] >> 16)


def _weight_row(K, code_at, scale=127):
    wc = np.zeros(K // 2, np.uint8)
    for k, c in code_at.items():
        k = int(k)
        wc[k // 2] |= np.uint8(c << (4 * (k % 2)))
    ws = np.full(K // 32, scale, np.uint8)
    return wc, ws


def _dequant_w(codes, scales):
    """Independent dequantisation: nibble k of byte k//2 (low nibble first) times 2^(s-127)."""
    lo = codes & 15
    hi = codes >> 4
    n = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    vals = E2M1_SPEC[n]
    return vals * np.exp2(np.repeat(scales.astype(np.float64) - 127, 32, axis=-1))


def _dequant_x(lay):
    if lay["kind"] == synth.ACT_BF16:
        return torch.from_numpy(lay["x"].view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    x = torch.from_numpy(lay["x"]).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return x * np.exp2(np.repeat(lay["sx"].astype(np.float64) - 127, 32, axis=-1))


def _bf16_value(b):
    return float(np.array([int(b) << 16], np.uint32).view(np.float32)[0])


def nearest_bf16(v):
    """The bf16 value nearest to the float64 v, ties to the even code, found by search over the
    codes next to binary32(v)'s truncation (an independent restatement of round-to-nearest)."""
    if math.isnan(v) or math.isinf(v) or v == 0.0:
        return v
    if abs(v) >= 2.0 ** 128 - 2.0 ** 119:
        return math.copysign(math.inf, v)
    b0 = int(np.array([v], np.float32).view(np.uint32)[0] >> 16) & 0x7FFF
    sign = 0x8000 if v < 0 else 0
    best = None
    for b in range(max(0, b0 - 2), min(0x7F7F, b0 + 2) + 1):
        c = _bf16_value(sign | b)
        key = (abs(v - c), b & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]



@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden_chain_order(orc, case):
    K = case["K"]
    wc, ws = _weight_row(K, case["w_code_at"], case.get("w_scale", 127))
    xc = np.zeros(K, np.float32)
    for k, v in case["x_bf16_at"].items():
        xc[int(k)] = np.float32(v)
    got = orc.chain_dot(wc, ws, xc, np.ones(K // 32, np.float32))
    assert got == case["expected"]
    if "expected_sign_negative" in case:
        assert (math.copysign(1, got) < 0) == case["expected_sign_negative"]


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["combine_cases"], ids=lambda c: c["name"])
def test_golden_combine(orc, case):
    d = np.array(case["d"], np.float32)[:, None]
    w = np.array(case["w"], np.float32)
    yb, yf = orc.combine_chain(d, w)
    assert yf[0] == np.float32(case["expected_f32"])
    assert yb[0] == orc.f32_to_bf16(np.array([case["expected_f32"]], np.float32))[0]


def _tiny_layer(kind=synth.ACT_BF16, R=4, seed=11):
    cfg = synth.workload("tiny", kind=kind, seed=seed)
    return synth.make_layer_numpy(cfg, R=R)


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16])
def test_one_hot_reads_one_weight(orc, kind):
    """x = e_i (value 1 at index i, scale 2^0): g_n equals the dequantised weight W[n, i]
    exactly; i sweeps both nibbles of a byte and both sides of a group boundary."""
    lay = _tiny_layer(kind)
    H, I = lay["H"], lay["I"]
    for i in [0, 1, 30, 31, 32, 33, 63, 64, H - 1]:
        if kind == synth.ACT_E4M3:
            x = np.zeros((1, H), np.uint8)
            x[0, i] = 0x38                          # E4M3 1.0
            sx = np.full((1, H // 32), 127, np.uint8)
        else:
            x = np.zeros((1, H), np.uint16)
            x[0, i] = _bf16_bits(1.0)
            sx = None
        one = dict(lay, x=x, sx=sx, ids=np.array([[3, 5]], np.int32), w=np.ones((1, 2), np.float32))
        ref_g = _dequant_w(lay["wg"][3], lay["sg"][3])[:, i]
        ref_u = _dequant_w(lay["wu"][5], lay["su"][5])[:, i]
        c = orc.layer_chain(one)
        f = orc.layer_f64(one)
        assert np.array_equal(c["g"][0, 0].astype(np.float64), ref_g)
        assert np.array_equal(c["u"][0, 1].astype(np.float64), ref_u)
        assert np.array_equal(f["g"][0, 0], ref_g)


def test_exact_integer_sums(orc):
    """All weights 1.0 at scale 2^0 and small-integer activations: the chain is the exact sum."""
    rng = np.random.default_rng(3)
    K = 1024
    wc = np.full(K // 2, 0x22, np.uint8)
    ws = np.full(K // 32, 127, np.uint8)
    xi = rng.integers(-15, 16, size=K)
    got = orc.chain_dot(wc, ws, xi.astype(np.float32), np.ones(K // 32, np.float32))
    assert got == float(xi.sum())


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16])
def test_f64_matches_torch_float64_matmul(orc, kind):
    lay = _tiny_layer(kind)
    f = orc.layer_f64(lay)
    xh = _dequant_x(lay)
    rt = orc.route(lay["ids"], lay["E"])
    for p in range(len(rt["pair_row"])):
        r, j = int(rt["pair_row"][p]), int(rt["pair_slot"][p])
        e = int(lay["ids"][r, j])
        Wg = torch.from_numpy(_dequant_w(lay["wg"][e], lay["sg"][e]))
        Wu = torch.from_numpy(_dequant_w(lay["wu"][e], lay["su"][e]))
        x = torch.from_numpy(xh[r])
        g = (Wg @ x).numpy()
        u = (Wu @ x).numpy()
        assert np.all(np.abs(f["g"][r, j] - g) <= 1e-12 * f["mg"][r, j] + 1e-300)
        assert np.all(np.abs(f["u"][r, j] - u) <= 1e-12 * f["mu"][r, j] + 1e-300)
        # down from the oracle's own quantised h, dequantised here independently
        if kind == synth.ACT_E4M3:
            q, s = orc.quant_e4m3_f64(f["h"][r, j])
            hh = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy() * np.exp2(np.repeat(s.astype(np.float64) - 127, 32))
        else:
            hh = np.array([nearest_bf16(v) for v in f["h"][r, j]])  # h rounded once from float64
        Wd = torch.from_numpy(_dequant_w(lay["wd"][e], lay["sd"][e]))
        d = (Wd @ torch.from_numpy(hh)).numpy()
        assert np.all(np.abs(f["d"][r, j] - d) <= 1e-12 * f["md"][r, j] + 1e-300)
    # combine: y = sum_j w_j d_j
    for r in range(lay["ids"].shape[0]):
        y = (lay["w"][r].astype(np.float64)[:, None] * f["d"][r]).sum(axis=0)
        assert np.all(np.abs(f["y"][r] - y) <= 1e-12 * f["my"][r] + 1e-300)
    # silu * u in float64 against torch
    h = (torch.nn.functional.silu(torch.from_numpy(f["g"])) * torch.from_numpy(f["u"])).numpy()
    assert np.all(np.abs(f["h"] - h) <= 1e-12 * f["mh"] + 1e-300)


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16])
def test_chain_within_f64_bound(orc, kind):
    cfg = synth.workload("tiny", kind=kind, H=1024, I=256, E=16, k=4, seed=21)
    lay = synth.make_layer_numpy(cfg, R=6)
    c = orc.layer_chain(lay)
    rt = c["route"]
    h_in = {(int(r), int(j)): (c["hq"][r, j], c["hs"][r, j] if kind == synth.ACT_E4M3 else None)
            for r, j in zip(rt["pair_row"], rt["pair_slot"])}
    f = orc.layer_f64(lay, h_in=h_in)
    mask = np.zeros(lay["ids"].shape, bool)
    mask[rt["pair_row"], rt["pair_slot"]] = True
    for name in ("g", "u", "h", "d"):
        ok = orc.within_tol(c[name][mask], f[name][mask], f["m" + name][mask])
        assert ok.all(), name
    assert orc.within_tol(c["y_f32"], f["y"], f["my"]).all()
    # and the error is real but small: the chain is not the float64 sum bit for bit
    assert np.abs(c["g"][mask] - f["g"][mask]).max() > 0


def test_epilogue_special_values(orc):
    g = np.array([0.0, -0.0, -100.0, 100.0, 1.0], np.float32)
    u = np.array([3.0, 3.0, 2.0, 2.0, -1.0], np.float32)
    h = orc.silu_mul(g, u)
    assert h[0] == 0.0 and h[1] == 0.0
    assert h[2] == 0.0 and math.copysign(1, h[2]) < 0      # exp(100) overflows: g / inf = -0
    assert h[3] == np.float32(200.0)
    ref = float(torch.nn.functional.silu(torch.tensor(1.0, dtype=torch.float64))) * -1.0
    assert abs(h[4] - ref) <= 2 ** -22


def test_combine_unit_weight_is_bf16_rounding(orc):
    rng = np.random.default_rng(9)
    d = rng.standard_normal((1, 4096)).astype(np.float32)
    yb, yf = orc.combine_chain(d, np.ones(1, np.float32))
    assert np.array_equal(yf, d[0])
    ref = torch.from_numpy(d[0].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(yb, ref)


def test_combine_power_of_two_weights_exact(orc):
    rng = np.random.default_rng(10)
    d = rng.integers(-100, 100, size=(8, 512)).astype(np.float32)
    w = np.exp2(rng.integers(-3, 3, size=8)).astype(np.float32)
    _, yf = orc.combine_chain(d, w)
    assert np.array_equal(yf.astype(np.float64), (w.astype(np.float64)[:, None] * d).sum(axis=0))
