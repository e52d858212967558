"""Pins of the oracle's routing (expert-major row lists) by brute force against an
independent formulation: sort the valid (expert, row, slot) triples."""
import numpy as np
import pytest


def _brute(ids, E):
    R, k = ids.shape
    trip = []
    status = 0
    for r in range(R):
        seen = set()
        for j in range(k):
            e = int(ids[r, j])
            if not 0 <= e < E:
                status |= 1
                continue
            if e in seen:
                status |= 2
                continue
            seen.add(e)
            trip.append((e, r, j))
    trip.sort()
    offs = np.zeros(E + 1, np.int64)
    for e, _, _ in trip:
        offs[e + 1] += 1
    offs = np.cumsum(offs)
    active = sorted(set(e for e, _, _ in trip))
    return status, offs, [t[1] for t in trip], [t[2] for t in trip], active


@pytest.mark.parametrize("seed", range(40))
def test_route_matches_sorted_triples(orc, seed):
    rng = np.random.default_rng(seed)
    E = int(rng.choice([4, 8, 33, 256]))
    k = int(rng.integers(1, min(E, 9)))
    R = int(rng.integers(0, 40))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(R)]) if R else np.zeros((0, k), np.int64)
    if seed % 3 == 0 and R:   # plant out-of-range ids and duplicates
        ids[rng.integers(0, R), rng.integers(0, k)] = rng.choice([-1, E, E + 5])
        if k > 1:
            r = rng.integers(0, R)
            ids[r, k - 1] = ids[r, 0]
    ids = ids.astype(np.int32).reshape(R, k)
    got = orc.route(ids, E)
    st, offs, prow, pslot, active = _brute(ids, E)
    assert got["status"] == st
    assert np.array_equal(got["offs"], offs)
    assert list(got["pair_row"]) == prow and list(got["pair_slot"]) == pslot
    assert list(got["active"]) == active and got["n_active"] == len(active)


def test_route_ten_thousand_small_random_cases(orc):
    # many small routings with out-of-range ids and repeats drawn freely (not only planted)
    rng = np.random.default_rng(2024)
    for _ in range(10000):
        E = int(rng.integers(1, 17))
        k = int(rng.integers(1, min(E, 4) + 1))
        R = int(rng.integers(0, 13))
        ids = rng.integers(-2, E + 2, size=(R, k)).astype(np.int32)
        got = orc.route(ids, E)
        st, offs, prow, pslot, active = _brute(ids, E)
        assert got["status"] == st
        assert np.array_equal(got["offs"], offs)
        assert list(got["pair_row"]) == prow and list(got["pair_slot"]) == pslot
        assert list(got["active"]) == active and got["n_active"] == len(active)
