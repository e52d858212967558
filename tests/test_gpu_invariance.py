"""Row invariance on the GPU (the equality probe of TensorFold PR #2983, "Kernel contract"):
a launch's activations (h), outputs (d) and combine output (y) are bit-equal to each row
launched alone, under same, disjoint and random routing at R = 1, 2, 3, 4, 5, 7, 8, 9, 16,
finite and with NaN/Inf planted in one row (54 cases a format). Also: the pass-size knobs
change no bit; permuting the rows permutes the outputs; padding rows and left-out pairs are
never written."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import gpu_util as gu  # noqa: E402
from moe_routed_expert_major_gb300 import tfx  # noqa: E402

H, I, E, K = 1024, 256, 64, 4
ROWS = [1, 2, 3, 4, 5, 7, 8, 9, 16]


@pytest.fixture(scope="module")
def weights():
    from moe_routed_expert_major_gb300 import build
    build.build()
    tfx.load()
    lay = synth.make_layer_numpy(synth.workload("tiny", kind=synth.ACT_E4M3, H=H, I=I, E=E, k=K, seed=99), R=1)
    d = tfx.dims(H, I, E, K)
    return lay, gu.pack(d, gu.device_weights_from_numpy(lay))


def make_case(base, kind, routing, R, planted, seed):
    rng = np.random.default_rng(seed)
    lay = {n: base[n] for n in ("H", "I", "E", "k", "wg", "sg", "wu", "su", "wd", "sd")}
    lay["kind"] = kind
    z = rng.standard_normal((R, H)).astype(np.float32)
    lay["x"], lay["sx"] = synth.activations(z, kind)
    if routing == "same":
        ex = rng.choice(E, size=K, replace=False)
        ids = np.stack([rng.permutation(ex) for _ in range(R)])
    elif routing == "disjoint":
        perm = rng.permutation(E)
        ids = np.stack([rng.permutation(perm[K * r:K * r + K]) for r in range(R)])
    else:
        ids = np.stack([rng.permutation(E)[:K] for _ in range(R)])
    lay["ids"] = ids.astype(np.int32)
    lay["w"] = rng.dirichlet(np.ones(K), size=R).astype(np.float32)
    if planted:
        synth.plant_nonfinite(lay, R // 2, seed=seed)
    return lay


def row_view(lay, r):
    one = dict(lay)
    one["x"] = lay["x"][r:r + 1].copy()
    one["sx"] = None if lay["sx"] is None else lay["sx"][r:r + 1].copy()
    one["ids"] = lay["ids"][r:r + 1].copy()
    one["w"] = lay["w"][r:r + 1].copy()
    return one


def outputs_by_row(lay, res):
    h = gu.per_pair(res, "h", lay)
    hs = gu.per_pair(res, "h_scale", lay) if lay["kind"] == synth.ACT_E4M3 else None
    return h, hs, res["out"][:lay["ids"].shape[0]], res["y"][:lay["ids"].shape[0]]


def assert_rows_equal(a, b, ra, rb):
    ha, hsa, da, ya = a
    hb, hsb, db, yb = b
    assert np.array_equal(ha[ra].view(np.uint8), hb[rb].view(np.uint8)), "act differs"
    if hsa is not None:
        assert np.array_equal(hsa[ra], hsb[rb]), "act scale differs"
    assert np.array_equal(da[ra].view(np.uint32), db[rb].view(np.uint32)), "out differs"
    assert np.array_equal(ya[ra].view(np.uint16), yb[rb].view(np.uint16)), "combine output differs"


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16], ids=["e4m3", "bf16"])
@pytest.mark.parametrize("planted", [False, True], ids=["finite", "nan_inf"])
@pytest.mark.parametrize("routing", ["same", "disjoint", "random"])
def test_rows_equal_alone(weights, kind, routing, planted):
    base, packed = weights
    for R in ROWS:
        lay = make_case(base, kind, routing, R, planted, seed=1000 + R)
        res = gu.run_layer(lay, packed, debug=False)
        assert res["status"] == 0
        full = outputs_by_row(lay, res)
        for r in range(R):
            one = row_view(lay, r)
            alone = outputs_by_row(one, gu.run_layer(one, packed, debug=False))
            assert_rows_equal(full, alone, r, 0)
        if planted:
            pr = R // 2
            y = (full[3][pr].view(np.uint16).astype(np.uint32) << 16).view(np.float32)
            assert np.isnan(y).any(), "planted NaN/Inf did not reach its row"
            clean = make_case(base, kind, routing, R, False, seed=1000 + R)
            cres = outputs_by_row(clean, gu.run_layer(clean, packed, debug=False))
            for r in range(R):
                if r != pr:
                    assert_rows_equal(full, cres, r, r)
                    yr = (full[3][r].view(np.uint16).astype(np.uint32) << 16).view(np.float32)
                    assert np.isfinite(yr).all()


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16], ids=["e4m3", "bf16"])
def test_pass_size_changes_no_bit(weights, kind):
    base, packed = weights
    for routing, R in (("same", 16), ("same", 5), ("random", 16), ("same", 3)):
        lay = make_case(base, kind, routing, R, False, seed=7 + R)
        ref = outputs_by_row(lay, gu.run_layer(lay, packed, debug=False))
        for mp in (1, 2, 3, 4, 5, 6, 7, 8):
            for tm in (0, 1, 2):
                ou = tfx.opts_struct(max_pass=mp, tier_mode=tm)
                od = tfx.opts_struct(max_pass=min(mp, 4), tier_mode=tm)
                got = outputs_by_row(lay, gu.run_layer(lay, packed, debug=False, opts_upc=ou, opts_down=od))
                for r in range(R):
                    assert_rows_equal(ref, got, r, r)


def test_row_permutation(weights):
    base, packed = weights
    lay = make_case(base, synth.ACT_E4M3, "random", 16, True, seed=5)
    ref = outputs_by_row(lay, gu.run_layer(lay, packed, debug=False))
    perm = np.random.default_rng(5).permutation(16)
    pl = dict(lay)
    pl["x"], pl["sx"], pl["ids"], pl["w"] = lay["x"][perm].copy(), lay["sx"][perm].copy(), lay["ids"][perm].copy(), lay["w"][perm].copy()
    got = outputs_by_row(pl, gu.run_layer(pl, packed, debug=False))
    for i, r in enumerate(perm):
        assert_rows_equal(ref, got, r, i)


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16], ids=["e4m3", "bf16"])
def test_padding_rows_never_written(weights, kind):
    """Every pass at 8 rows with 3 real rows: the 5 padding rows of the last expert would land
    past the used pairs; those bytes, and the left-out pair's outputs, keep their canary."""
    base, packed = weights
    lay = make_case(base, kind, "same", 3, False, seed=11)
    lay["ids"][2, 3] = E + 1                       # one left-out pair: 11 pairs used of 12
    ou = tfx.opts_struct(max_pass=8, tier_mode=1)
    od = tfx.opts_struct(max_pass=4, tier_mode=1)
    res = gu.run_layer(lay, packed, debug=True, opts_upc=ou, opts_down=od, canary=0x5A)
    assert res["status"] == tfx.ST_RANGE
    used = int(res["route"]["offs"][-1])
    assert used == 11
    assert np.all(res["h"][used:].view(np.uint8) == 0x5A)
    if res["h_scale"] is not None:
        assert np.all(res["h_scale"][used:] == 0x5A)
    assert np.all(res["gu_dbg"][used:].view(np.uint8) == 0x5A)
    assert np.all(res["h_dbg"][used:].view(np.uint8) == 0x5A)
    assert np.all(res["out"][2, 3].view(np.uint8) == 0x5A)
    # and the written rows equal the default launch
    ref = outputs_by_row(lay, gu.run_layer(lay, packed, debug=False))
    got = outputs_by_row(lay, res)
    for r in range(2):
        assert_rows_equal(ref, got, r, r)
