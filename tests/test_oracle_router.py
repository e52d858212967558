"""Pins of the oracle's router (top-k from logits): closed-form weights, the tie and NaN
order, properties of the selection checked against the definition on random rows."""
import json
import math
import os

import numpy as np
import pytest

import oracle


def test_equal_logits_take_the_lowest_ids_with_equal_weights():
    for mode in (0, 1):
        ids, w = oracle.router(np.zeros((2, 10), np.float32), 4, mode)
        assert ids.tolist() == [[0, 1, 2, 3]] * 2
        assert np.all(w == 0.25)


def test_powers_of_two_weights():
    # logits c - j*ln2 on a shuffled set of experts: softmax weights 2^-j / (2 - 2^(1-k))
    rng = np.random.default_rng(5)
    k, n = 5, 32
    experts = rng.permutation(n)[:k]
    row = np.full(n, -1e4)
    for j, e in enumerate(experts):
        row[e] = 3.0 - j * math.log(2.0)
    ids, w = oracle.router(row[None, :], k, 0)
    assert ids[0].tolist() == experts.tolist()
    want = np.array([2.0 ** -j for j in range(k)])
    want /= want.sum()
    assert np.allclose(w[0], want, rtol=1e-12, atol=0)


def test_sigmoid_closed_form():
    row = np.array([[0.0, math.log(3.0), -math.log(3.0), -50.0]])
    ids, w = oracle.router(row, 3, 1)
    assert ids[0].tolist() == [1, 0, 2]
    t = np.array([0.75, 0.5, 0.25])  # 1 / (1 + e^-l) at ln 3, 0, -ln 3
    assert np.allclose(w[0], t / t.sum(), rtol=1e-12, atol=0)


def test_ties_signed_zero_and_nan_order():
    nan = float("nan")
    row = np.array([[1.0, nan, -0.0, 0.0, 1.0, -np.inf, nan]])
    ids, _ = oracle.router(row, 7, 0)
    # numbers in descending order, equal values by id (-0 == +0), then NaNs by id
    assert ids[0].tolist() == [0, 4, 2, 3, 5, 1, 6]


def test_shift_invariance_and_shared_slot():
    rng = np.random.default_rng(9)
    L = rng.standard_normal((6, 40))
    ids0, w0 = oracle.router(L, 8, 0)
    ids1, w1 = oracle.router(L + 12.5, 8, 0, shared=40)
    assert np.array_equal(ids1[:, :8], ids0) and np.all(ids1[:, 8] == 40)
    assert np.all(w1[:, 8] == 1.0)
    assert np.allclose(w1[:, :8], w0, rtol=1e-12, atol=0)


@pytest.mark.parametrize("mode", [0, 1])
def test_selection_matches_the_definition_on_random_rows(mode):
    rng = np.random.default_rng(13)
    L = np.round(rng.standard_normal((50, 24)) * 2) / 2  # many equal values
    k = 6
    ids, w = oracle.router(L, k, mode)
    for r in range(L.shape[0]):
        sel = list(ids[r])
        rest = [e for e in range(L.shape[1]) if e not in sel]
        assert len(set(sel)) == k
        # every selected logit >= every unselected one; an equal unselected one has a larger id
        for e in sel:
            for f in rest:
                assert L[r, e] > L[r, f] or (L[r, e] == L[r, f] and e < f)
        # slots in descending order, equal values by id
        for a, b in zip(sel, sel[1:]):
            assert L[r, a] > L[r, b] or (L[r, a] == L[r, b] and a < b)
        assert abs(w[r].sum() - 1.0) < 1e-12 and np.all(w[r] > 0)
        if mode == 0:  # weight ratios are exp of logit differences
            assert np.allclose(w[r][1:] / w[r][0], np.exp(L[r, sel[1:]] - L[r, sel[0]]), rtol=1e-12)


# ------------------------------------------------------------------ group-limited routing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "router_grouped.json")


def _bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def test_sigmoid32_error_bound_and_special_values():
    l = np.linspace(-85.0, 85.0, 400001).astype(np.float32)
    s = oracle.sigmoid32(l).astype(np.float64)
    exact = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    assert np.max(np.abs(s - exact) / exact) < 4 * 2.0 ** -24
    # symmetry: s(l) + s(-l) = 1 up to the roundings of the two values
    assert np.max(np.abs(oracle.sigmoid32(l).astype(np.float64) + oracle.sigmoid32(-l) - 1.0)) <= 2.0 ** -23
    sp = oracle.sigmoid32(np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -100.0, -86.0], np.float32))
    assert sp[0] == 0.5 and sp[1] == 0.5 and sp[2] == 1.0 and np.isnan(sp[4])
    # below -86 the argument is taken as -86: a positive normal number near e^-86
    assert sp[3] == sp[5] == sp[6] and np.float32(1.17e-38) < sp[6] and abs(sp[6] / math.exp(-86.0) - 1.0) < 1e-6
    # the Cody-Waite head is exact times any |n| < 128 and head + tail is ln 2
    hi, lo = float(oracle._LN2_HI), float(oracle._LN2_LO)
    assert (hi * 2 ** 16).is_integer() and abs(hi + lo - math.log(2.0)) < 1e-12


def test_grouped_golden_cases():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        L = np.array([[float(v) for v in c["logits"]]], np.float32)
        b = None if c["bias"] is None else np.array(c["bias"], np.float32)
        ids, w = oracle.router_grouped(L, c["top_k"], c["n_group"], c["topk_group"], b, c["scale"])
        assert ids[0].tolist() == c["ids"], c["name"]
        assert [int(v, 16) for v in c["w_bits"]] == _bits(w[0]).tolist(), c["name"]


def test_grouped_with_every_group_kept_is_plain_sigmoid_routing():
    # all groups kept and no bias: the choice is the top-k of the sigmoid, i.e. of the logits
    # (distinct, well-separated logits), and the weights are the normalised sigmoid in float64
    # within fp32 rounding
    rng = np.random.default_rng(21)
    L = (rng.permutation(64 * 30).reshape(30, 64) * 0.01 - 9.6).astype(np.float32)
    ids, w = oracle.router_grouped(L, 6, 8, 8, None, 2.5)
    ids0, w0 = oracle.router(L, 6, 1)
    assert np.array_equal(ids, ids0)
    assert np.allclose(w, 2.5 * w0, rtol=2e-6, atol=0)


def test_grouped_selection_properties_on_random_rows():
    rng = np.random.default_rng(22)
    n, ng, kg, k = 64, 8, 3, 6
    gs = n // ng
    L = (np.round(rng.standard_normal((40, n)) * 4) / 4).astype(np.float32)  # many equal values
    bias = (np.round(rng.standard_normal(n) * 8) / 64).astype(np.float32)
    ids, w = oracle.router_grouped(L, k, ng, kg, bias, 1.0)
    s = oracle.sigmoid32(L)
    c = (s + bias[None, :]).astype(np.float64)
    for r in range(L.shape[0]):
        G = np.array([np.sort(c[r, g * gs:(g + 1) * gs])[-2:].sum() for g in range(ng)])
        kept = sorted(set(int(e) // gs for e in ids[r]))
        assert len(kept) <= kg and len(set(ids[r].tolist())) == k
        # no dropped group scores above the weakest kept group that a selection could need
        full = np.argsort(-G, kind="stable")[:kg]
        assert set(kept) <= set(full.tolist())
        allowed = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in full])
        want = allowed[np.argsort(-c[r, allowed], kind="stable")[:k]]
        assert ids[r].tolist() == want.tolist()
        # weights: normalised sigmoid (not the biased score)
        assert np.allclose(w[r], s[r, ids[r]] / s[r, ids[r]].astype(np.float64).sum(), rtol=2e-6, atol=0)


def test_grouped_bias_steers_the_choice_not_the_weights_and_shared_slot():
    rng = np.random.default_rng(23)
    L = rng.standard_normal((8, 32)).astype(np.float32)
    bias = np.zeros(32, np.float32)
    bias[5] = 4.0  # expert 5 is always chosen
    ids, w = oracle.router_grouped(L, 4, 4, 2, bias, 1.0, shared=32)
    ids0, w0 = oracle.router_grouped(L, 4, 4, 2, None, 1.0)
    assert np.all(ids[:, 0] == 5) and np.all(ids[:, 4] == 32) and np.all(w[:, 4] == 1.0)
    s = oracle.sigmoid32(L)
    for r in range(8):
        t = s[r, ids[r, :4]]
        acc = np.float32(0.0)
        for v in t:
            acc = np.float32(acc + v)
        assert np.array_equal(_bits(w[r, :4]), _bits(t / acc))
        if 5 in ids0[r]:
            assert sorted(ids0[r].tolist()) == sorted(ids[r, :4].tolist())
