"""Pins of the oracle's router (top-k from logits): closed-form weights, the tie and NaN
order, properties of the selection checked against the definition on random rows."""
import math

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
