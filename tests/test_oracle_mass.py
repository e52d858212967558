"""Pins of the float64 mode's mass, the Σ|terms| that every value carries into the tolerance
|err| <= 1e-3 * mass + 1e-6 ("Receipt › Kernel contract" of "dsv41 metal: decode experts
decode an expert's weights once for all of its rows": each output is registered against the
float64 reference), and of the float64 mode's bf16 rounding of h.

- One output: closed forms. Equal and opposite terms (sum 0, mass K), one nonzero term,
  terms of one sign (mass = |sum|), whole-row and per-group power-of-two scales (mass scales
  by the same power), integer terms (mass = Σ|x|).
- SwiGLU: special points worked by hand; the first-order propagation against derivatives
  from torch autograd and against finite differences with the worst sign of each input's
  error.
- Combine: a hand case and Σ|w_j| mass_j on random values.
- The whole tiny layer: g, u, d and y masses against |W| @ |x| from an independent
  dequantisation and a library matmul.
- The tolerance test itself at its edge.
- bf16 rounding of a float64: one rounding, to nearest even, checked by hand cases where a
  binary32 step in between would give another answer, and on random values against the
  nearest bf16 found by search.
"""
import math

import numpy as np
import pytest
import torch

import synth
from test_oracle_chain import _dequant_w, _dequant_x, _weight_row, nearest_bf16

ONE = 0x2      # E2M1 code of +1.0
TWO = 0x4      # +2.0
M_THREE = 0xD  # -3.0


def _ones_row(K, code=ONE):
    return _weight_row(K, {k: code for k in range(K)})


# ---------------------------------------------------------------------------------- one output

def test_mass_of_cancelling_terms_is_k(orc):
    """Weights +1 and x = +1, -1, +1, ...: the sum is 0 and every term has magnitude 1."""
    K = 1024
    wc, ws = _ones_row(K)
    x = np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
    v, m = orc.f64_dot(wc, ws, x)
    assert v == 0.0 and m == float(K)


@pytest.mark.parametrize("i", [0, 1, 31, 32, 63, 200, 255])
def test_mass_of_one_term(orc, i):
    """One nonzero activation x_i = -3.5 against a random row: value W[i] * -3.5, mass |W[i]| * 3.5."""
    rng = np.random.default_rng(i)
    K = 256
    wc = rng.integers(0, 256, K // 2).astype(np.uint8)
    ws = rng.integers(123, 130, K // 32).astype(np.uint8)
    x = np.zeros(K)
    x[i] = -3.5
    wi = _dequant_w(wc[None], ws[None])[0, i]
    v, m = orc.f64_dot(wc, ws, x)
    assert v == wi * -3.5
    assert m == abs(wi) * 3.5


def test_mass_of_same_sign_terms_is_the_magnitude(orc):
    """Nonnegative weights against positive x: no cancellation, so the mass is |sum|."""
    rng = np.random.default_rng(1)
    K = 512
    wc = (rng.integers(0, 8, K // 2) | (rng.integers(0, 8, K // 2) << 4)).astype(np.uint8)  # sign bits clear
    ws = rng.integers(124, 129, K // 32).astype(np.uint8)
    x = rng.integers(1, 9, K).astype(np.float64) / 4.0
    v, m = orc.f64_dot(wc, ws, x)
    assert v > 0 and m == v
    # and with x negated, the value flips and the mass does not
    v2, m2 = orc.f64_dot(wc, ws, -x)
    assert v2 == -v and m2 == m


@pytest.mark.parametrize("s", [-5, -1, 1, 3])
def test_mass_scales_with_the_weight_scale(orc, s):
    """Every group's scale code raised by s multiplies the mass by 2^s exactly; one group's
    scale raised by s adds (2^s - 1) times that group's own mass."""
    rng = np.random.default_rng(10 + s)
    K = 256
    wc = rng.integers(0, 256, K // 2).astype(np.uint8)
    ws = np.full(K // 32, 127, np.uint8)
    x = rng.standard_normal(K)
    _, m0 = orc.f64_dot(wc, ws, x)
    _, m1 = orc.f64_dot(wc, ws + np.uint8(s) if s > 0 else ws - np.uint8(-s), x)
    assert m1 == math.ldexp(m0, s)
    g = 3
    xg = np.zeros(K)
    xg[32 * g:32 * g + 32] = x[32 * g:32 * g + 32]
    _, mg = orc.f64_dot(wc, ws, xg)
    ws2 = ws.copy()
    ws2[g] = 127 + s
    _, m2 = orc.f64_dot(wc, ws2, x)
    assert m2 == pytest.approx(m0 + (2.0 ** s - 1.0) * mg, rel=1e-14)


def test_mass_of_integer_terms(orc):
    """Weights +2 and -3 alternating by group against small integers: sum and Σ|terms| are
    exact integers."""
    rng = np.random.default_rng(2)
    K = 1024
    codes = {k: (TWO if (k // 32) % 2 == 0 else M_THREE) for k in range(K)}
    wc, ws = _weight_row(K, codes)
    x = rng.integers(-15, 16, K).astype(np.float64)
    w = np.where((np.arange(K) // 32) % 2 == 0, 2.0, -3.0)
    v, m = orc.f64_dot(wc, ws, x)
    assert v == float((w * x).sum()) and m == float(np.abs(w * x).sum())


# ---------------------------------------------------------------------------------- SwiGLU

def test_silu_mass_worked_points(orc):
    """h = silu(g) u with mass |silu'(g)| mg |u| + |silu(g)| mu + |h|, silu'(0) = 1/2:
    g = 0, u = 2, mg = 1, mu = 0 -> h = 0, mass 1;  g = 0, mu only -> mass 0 (silu(0) = 0);
    mg = mu = 0 -> mass |h| (the value's own rounding)."""
    h, mh = orc.silu_mul_f64([0.0, 0.0, 1.5], [2.0, 2.0, -4.0], [1.0, 0.0, 0.0], [0.0, 3.0, 0.0])
    assert h[0] == 0.0 and mh[0] == 1.0
    assert h[1] == 0.0 and mh[1] == 0.0
    assert mh[2] == abs(h[2]) and h[2] < 0


def _silu_grad(g, u):
    gt = torch.tensor(g, dtype=torch.float64, requires_grad=True)
    ut = torch.tensor(u, dtype=torch.float64, requires_grad=True)
    h = torch.nn.functional.silu(gt) * ut
    h.sum().backward()
    return h.detach().numpy(), gt.grad.numpy(), ut.grad.numpy()


def _points(n=400, seed=5):
    rng = np.random.default_rng(seed)
    g = np.concatenate([rng.standard_normal(n) * 4, [-30.0, -8.0, -1.278464542761074, 2.0, 30.0]])
    u = rng.standard_normal(g.size) * 3
    mg = np.abs(rng.standard_normal(g.size)) * 5 + np.abs(g)
    mu = np.abs(rng.standard_normal(g.size)) * 5 + np.abs(u)
    return g, u, mg, mu


def test_silu_mass_against_autograd(orc):
    """The propagated mass equals |dh/dg| mg + |dh/du| mu + |h| with the derivatives from
    torch autograd (silu'(g) at g = -1.2785, its minimum, included)."""
    g, u, mg, mu = _points()
    h, mh = orc.silu_mul_f64(g, u, mg, mu)
    hr, dg, du = _silu_grad(g, u)
    assert np.allclose(h, hr, rtol=1e-14, atol=0)
    ref = np.abs(dg) * mg + np.abs(du) * mu + np.abs(hr)
    assert np.allclose(mh, ref, rtol=1e-12, atol=1e-300)


def test_silu_mass_against_finite_differences(orc):
    """mass - |h| is the first-order change of h when g and u move by eps * mg and eps * mu
    with the worst signs: the largest |h(g + a eps mg, u + b eps mu) - h| / eps over a, b = +-1
    (central differences, eps = 1e-6)."""
    g, u, mg, mu = _points(seed=6)
    _, mh = orc.silu_mul_f64(g, u, mg, mu)

    def hf(gg, uu):
        return gg / (1.0 + np.exp(-gg)) * uu

    h0 = hf(g, u)
    eps = 1e-6
    best = np.zeros_like(g)
    for a in (1.0, -1.0):
        for b in (1.0, -1.0):
            d = (hf(g + a * eps * mg, u + b * eps * mu) - hf(g - a * eps * mg, u - b * eps * mu)) / (2 * eps)
            best = np.maximum(best, np.abs(d))
    assert np.allclose(mh - np.abs(h0), best, rtol=1e-5, atol=1e-9)


# ---------------------------------------------------------------------------------- combine

def test_combine_mass_worked_case(orc):
    """d = (1, -2), masses (3, 5), w = (0.5, -0.25): y = 0.5 + 0.5 = 1, mass 0.5*3 + 0.25*5 = 2.75."""
    y, my = orc.combine_f64(np.array([[1.0], [-2.0]]), np.array([[3.0], [5.0]]), np.array([0.5, -0.25], np.float32))
    assert y[0] == 1.0 and my[0] == 2.75


def test_combine_mass_random(orc):
    rng = np.random.default_rng(7)
    k, H = 8, 300
    d = rng.standard_normal((k, H))
    md = np.abs(d) + np.abs(rng.standard_normal((k, H)))
    w = rng.standard_normal(k).astype(np.float32)
    y, my = orc.combine_f64(d, md, w)
    wd = w.astype(np.float64)
    assert np.allclose(y, (wd[:, None] * d).sum(0), rtol=1e-14, atol=1e-15)
    assert np.allclose(my, (np.abs(wd)[:, None] * md).sum(0), rtol=1e-14, atol=0)
    assert np.all(my >= np.abs(y))


# ---------------------------------------------------------------------------------- whole layer

@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16])
def test_layer_masses_against_library_matmul(orc, kind):
    """mg = |Wg| @ |x|, mu = |Wu| @ |x|, md = |Wd| @ |h|, my = Σ_j |w_j| md_j, with the
    weights and activations dequantised here and the products summed by torch (float64)."""
    cfg = synth.workload("tiny", kind=kind, seed=31)
    lay = synth.make_layer_numpy(cfg, R=4)
    f = orc.layer_f64(lay)
    xh = np.abs(_dequant_x(lay))
    rt = orc.route(lay["ids"], lay["E"])
    for p in range(len(rt["pair_row"])):
        r, j = int(rt["pair_row"][p]), int(rt["pair_slot"][p])
        e = int(lay["ids"][r, j])
        Ag = torch.from_numpy(np.abs(_dequant_w(lay["wg"][e], lay["sg"][e])))
        Au = torch.from_numpy(np.abs(_dequant_w(lay["wu"][e], lay["su"][e])))
        x = torch.from_numpy(xh[r])
        assert np.allclose(f["mg"][r, j], (Ag @ x).numpy(), rtol=1e-13, atol=0)
        assert np.allclose(f["mu"][r, j], (Au @ x).numpy(), rtol=1e-13, atol=0)
        if kind == synth.ACT_E4M3:
            q, s = orc.quant_e4m3_f64(f["h"][r, j])
            hh = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy() * np.exp2(
                np.repeat(s.astype(np.float64) - 127, 32))
        else:
            hh = np.array([nearest_bf16(v) for v in f["h"][r, j]])
        Ad = torch.from_numpy(np.abs(_dequant_w(lay["wd"][e], lay["sd"][e])))
        assert np.allclose(f["md"][r, j], (Ad @ torch.from_numpy(np.abs(hh))).numpy(), rtol=1e-13, atol=0)
    for r in range(lay["ids"].shape[0]):
        my = (np.abs(lay["w"][r].astype(np.float64))[:, None] * f["md"][r]).sum(0)
        assert np.allclose(f["my"][r], my, rtol=1e-13, atol=0)


def test_within_tol_edges(orc):
    """|err| <= 1e-3 mass + 1e-6 (+ extra): exactly at the bound passes, just past it fails;
    NaN matches only NaN."""
    ref = np.array([0.0, 0.0, 0.0, np.nan, np.nan, 0.0])
    mass = np.array([2.0, 2.0, 0.0, 1.0, 1.0, 2.0])
    bound = 1e-3 * 2.0 + 1e-6
    got = np.array([bound, bound * (1 + 1e-9), 1e-6, np.nan, 0.0, bound + 0.25])
    ok = orc.within_tol(got, ref, mass, extra=np.array([0, 0, 0, 0, 0, 0.25]))
    assert ok.tolist() == [True, False, True, True, False, True]


# ---------------------------------------------------------------------------------- bf16 of a float64

def test_f64_to_bf16_single_rounding(orc):
    """1 + 2^-8 is a bf16 midpoint (between 1 and 1 + 2^-7). A float64 just above it, 1 + 2^-8 +
    2^-30, is nearer to 1 + 2^-7; through binary32 it would first land on the midpoint and then
    go to 1 (the even neighbour). Exact midpoints go to the even code."""
    v = np.array([1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8 + 2.0 ** -30),
                  1 + 2.0 ** -8 - 2.0 ** -30])
    got = orc.f64_to_bf16(v)
    assert got.tolist() == [0x3F81, 0x3F80, 0x3F82, 0xBF81, 0x3F80]
    assert orc.f32_to_bf16(v[:1].astype(np.float32))[0] == 0x3F80  # what the binary32 step would give


def test_f64_to_bf16_special_values(orc):
    v = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 2.0 ** 128 - 2.0 ** 119, 2.0 ** 128 - 2.0 ** 119 - 2.0 ** 80,
                  2.0 ** -133, 2.0 ** -134, 2.0 ** -134 + 2.0 ** -160, 3 * 2.0 ** -134, 1e-300])
    got = orc.f64_to_bf16(v).tolist()
    assert got[:4] == [0x0000, 0x8000, 0x7F80, 0xFF80]
    assert (got[4] & 0x7F80) == 0x7F80 and (got[4] & 0x7F) != 0
    assert got[5] == 0x7F80 and got[6] == 0x7F7F           # the overflow midpoint rounds up; below it, the largest finite
    assert got[7] == 0x0001 and got[8] == 0x0000           # smallest subnormal; half of it ties to even (zero)
    assert got[9] == 0x0001 and got[10] == 0x0002 and got[11] == 0x0000


def test_f64_to_bf16_random_against_search(orc):
    rng = np.random.default_rng(12)
    v = rng.standard_normal(20000) * np.exp2(rng.integers(-140, 128, 20000).astype(np.float64))
    v = np.concatenate([v, rng.standard_normal(2000) * 2.0 ** -130])
    got = orc.f64_to_bf16(v)
    vals = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = np.array([nearest_bf16(t) for t in v])
    assert np.array_equal(vals, ref)
