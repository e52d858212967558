"""GPU parity of the chunk path (tfx_xp_upc_chunk / tfx_xp_down_chunk): block-scaled
tensor-core contractions that do not follow the fp32 chain, checked through the C ABI
against the oracle:
  * g, u, h (before quantisation), d and y within |err| <= 1e-3 * mass + 1e-6 of float64
    (d and y from the device's own quantised h, as for the rows path);
  * h's E4M3 codes and scales equal to the oracle's quantiser applied to the device's h;
  * the combine bit-equal to the oracle's slot-order chain over the device's d;
  * chunk invariance: every pair's h, d and y bits are the same whether its row runs alone
    or in chunks of 7, 64, 100 or 300 rows (experts then hold from one to two 128-pair
    tiles, so a pair moves between lanes and tiles);
  * the 4,096-row prompt chunk at full widths, in the launch configuration the benchmark
    times, on sampled rows."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import gpu_util as gu  # noqa: E402
from moe_routed_expert_major_gb300 import tfx  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_routed_expert_major_gb300 import build
    build.build()
    tfx.load()


def _worst(got, ref, mass):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(got) & np.isfinite(ref)
    if not fin.any():
        return 0.0
    return float(np.max(np.abs(got - ref)[fin] / (np.asarray(mass)[fin] + 1e-300)))


def check_chunk(orc, lay, res, rows=None):
    R, k = lay["ids"].shape
    kind = lay["kind"]
    assert res["status"] & ~(tfx.ST_RANGE | tfx.ST_DUP) == 0, res["status"]
    rt_o = orc.route(lay["ids"], lay["E"])
    n = int(rt_o["offs"][-1])
    rt = res["route"]
    assert np.array_equal(rt["offs"], rt_o["offs"])
    assert np.array_equal(rt["pair_row"][:n], rt_o["pair_row"]) and np.array_equal(rt["pair_slot"][:n], rt_o["pair_slot"])
    h_in = gu.h_in_from_gpu(lay, res)
    f = orc.layer_f64(lay, h_in=h_in, rows=rows)
    mask = np.zeros((R, k), bool)
    mask[rt_o["pair_row"], rt_o["pair_slot"]] = True
    if rows is not None:
        keep = np.zeros(R, bool)
        keep[list(rows)] = True
        mask &= keep[:, None]
    gud = gu.per_pair(res, "gu_dbg", lay)
    hd = gu.per_pair(res, "h_dbg", lay)
    for name, got, ref, mass in (("g", gud[:, :, 0][mask], f["g"][mask], f["mg"][mask]),
                                 ("u", gud[:, :, 1][mask], f["u"][mask], f["mu"][mask]),
                                 ("h", hd[mask], f["h"][mask], f["mh"][mask]),
                                 ("d", res["out"][mask], f["d"][mask], f["md"][mask])):
        ok = orc.within_tol(got, ref, mass)
        assert ok.all(), "%s: %d of %d outside the bound; worst |err|/mass = %.3g" % (
            name, int((~ok).sum()), ok.size, _worst(got, ref, mass))
    for p in range(n):
        r, j = int(rt_o["pair_row"][p]), int(rt_o["pair_slot"][p])
        if not mask[r, j]:
            continue
        q, s = orc.quantize_act(kind, res["h_dbg"][p])
        assert np.array_equal(res["h"][p], q) and np.array_equal(res["h_scale"][p], s), (r, j)
    for r in (range(R) if rows is None else rows):
        if not mask[r].all():
            continue
        yb_c, yf_c = orc.combine_chain(res["out"][r], lay["w"][r])
        assert gu.bits_equal(res["y_f32"][r], yf_c)
        assert gu.bf16_equal(res["y"][r].view(np.uint16), yb_c)
        yb = orc.bf16_to_f32(res["y"][r].view(np.uint16)).astype(np.float64)
        half_ulp = np.abs(f["y"][r]) * 2.0 ** -8
        assert orc.within_tol(yb, f["y"][r], f["my"][r], extra=half_ulp).all()


def _layer(H, I, E, k, R, seed):
    cfg = synth.workload("chunk", H=H, I=I, E=E, k=k, seed=seed)
    return synth.make_layer_numpy(cfg, R=R)


def _packed(lay):
    d = tfx.dims(lay["H"], lay["I"], lay["E"], lay["ids"].shape[1])
    return gu.pack(d, gu.device_weights_from_numpy(lay))


@pytest.mark.parametrize("H,I,E,k,R,seed", [
    (512, 512, 8, 2, 40, 11),      # small: one tile per expert
    (512, 512, 2, 2, 200, 12),     # 200 pairs per expert: two 128-pair tiles, ragged second
    (1024, 512, 4, 2, 300, 13),    # several weight-row tiles and k stages
])
def test_chunk_within_float64_bound(orc, H, I, E, k, R, seed):
    lay = _layer(H, I, E, k, R, seed)
    res = gu.run_layer_chunk(lay, _packed(lay))
    assert res["status"] == 0
    check_chunk(orc, lay, res)


def test_chunk_padding_rows_never_written():
    """Canaries in the buffers of pairs beyond the routed ones survive (lanes past a tile's
    real pairs are computed and dropped)."""
    lay = _layer(512, 512, 2, 2, 70, 14)
    res = gu.run_layer_chunk(lay, _packed(lay), canary=0x5A)
    n = int(res["route"]["offs"][-1])
    assert n == 140
    assert res["status"] == 0
    # h, h_scale and the debug rows are [R*k] sized: every row is a real pair here, so check
    # a launch with a left-out pair instead
    bad = dict(lay)
    bad["ids"] = lay["ids"].copy()
    bad["ids"][3, 1] = lay["E"] + 7  # out of range: left out
    res = gu.run_layer_chunk(bad, _packed(lay), canary=0x5A)
    assert res["status"] & tfx.ST_RANGE
    assert int(res["route"]["offs"][-1]) == 139
    assert np.all(res["h"][139].view(np.uint8) == 0x5A)
    assert np.all(res["h_scale"][139] == 0x5A)
    assert np.all(res["out"][3, 1].view(np.uint8) == 0x5A)


def _slice(lay, r0, r1):
    s = dict(lay)
    s["x"], s["sx"], s["ids"], s["w"] = lay["x"][r0:r1], lay["sx"][r0:r1], lay["ids"][r0:r1], lay["w"][r0:r1]
    return s


def _chunked(lay, packed, size):
    R, k = lay["ids"].shape
    hq, hsc, out, y = {}, {}, np.zeros((R, k, lay["H"]), np.float32), np.zeros((R, lay["H"]), np.int16)
    for r0 in range(0, R, size):
        r1 = min(R, r0 + size)
        res = gu.run_layer_chunk(_slice(lay, r0, r1), packed, debug=False)
        assert res["status"] == 0
        rt = res["route"]
        for p in range(int(rt["offs"][-1])):
            key = (r0 + int(rt["pair_row"][p]), int(rt["pair_slot"][p]))
            hq[key] = res["h"][p].copy()
            hsc[key] = res["h_scale"][p].copy()
        out[r0:r1] = res["out"][:r1 - r0]
        y[r0:r1] = res["y"][:r1 - r0]
    return hq, hsc, out, y


@pytest.mark.parametrize("H,I,E,k", [(2048, 512, 8, 4), (7168, 2048, 256, 8)])
def test_chunk_invariance(H, I, E, k):
    """Rows in chunks of 1, 7, 100 and 300 against 64-row chunks: identical bits."""
    R = 300
    cfg = synth.workload("chunk", H=H, I=I, E=E, k=k, seed=21)
    if E == 256:
        lay, dw = gu.full_layer(cfg, R=R)
        packed = gu.pack(tfx.dims(H, I, E, k), dw)
        sizes = [300, 100, 7]
    else:
        lay = synth.make_layer_numpy(cfg, R=R)
        packed = _packed(lay)
        sizes = [300, 100, 7, 1]
    ref = _chunked(lay, packed, 64)
    for size in sizes:
        got = _chunked(lay, packed, size)
        assert got[0].keys() == ref[0].keys()
        for key in ref[0]:
            assert np.array_equal(got[0][key], ref[0][key]), (size, key)
            assert np.array_equal(got[1][key], ref[1][key]), (size, key)
            r, j = key
            assert np.array_equal(got[2][r, j].view(np.uint32), ref[2][r, j].view(np.uint32)), (size, key)
        assert np.array_equal(got[3].view(np.uint16), ref[3].view(np.uint16)), size


def test_prompt_chunk_full_size_sampled(orc):
    """The 4,096-row chunk at H 7168, I 2048, E 256, top-8 (about 128 pairs per expert):
    sampled rows within the float64 bound, and rows alone give the same bits."""
    cfg = synth.workload("chunk")
    lay, dw = gu.full_layer(cfg)
    packed = gu.pack(tfx.dims(cfg["H"], cfg["I"], cfg["E"], cfg["k"]), dw)
    res = gu.run_layer_chunk(lay, packed)
    assert res["status"] == 0
    counts = np.diff(res["route"]["offs"])
    assert counts.max() > 128  # some experts span two tiles
    rows = [0, 1777, 4095]
    check_chunk(orc, lay, res, rows=rows)
    for r in (0, 4095):
        alone = gu.run_layer_chunk(_slice(lay, r, r + 1), packed, debug=False)
        assert np.array_equal(alone["out"][0].view(np.uint32), res["out"][r].view(np.uint32)), r
        assert np.array_equal(alone["y"][0].view(np.uint16), res["y"][r].view(np.uint16)), r
