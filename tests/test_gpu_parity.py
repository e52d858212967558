"""GPU parity against the oracle, through the C ABI: routing bit-exact; g, u, d and the
combine bit-exact against the fp32-chain oracle (d from the device's own quantised h);
h within the float64 bound and its quantisation equal to the oracle's quantiser applied to
the device's fp32 h; every final value within |err| <= 1e-3 * mass + 1e-6 of float64."""
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


def small_layer(kind, H=256, I=128, E=8, k=2, R=4, seed=1, routing="random"):
    cfg = synth.workload("tiny", kind=kind, H=H, I=I, E=E, k=k, seed=seed, routing=routing)
    return synth.make_layer_numpy(cfg, R=R)


def check_layer(orc, lay, res, rows=None):
    R, k = lay["ids"].shape
    kind = lay["kind"]
    assert res["status"] & ~(tfx.ST_RANGE | tfx.ST_DUP) == 0, res["status"]
    rt_o = orc.route(lay["ids"], lay["E"])
    n = int(rt_o["offs"][-1])
    rt = res["route"]
    assert np.array_equal(rt["offs"], rt_o["offs"])
    assert np.array_equal(rt["pair_row"][:n], rt_o["pair_row"]) and np.array_equal(rt["pair_slot"][:n], rt_o["pair_slot"])
    assert int(rt["n_active"][0]) == rt_o["n_active"]
    assert np.array_equal(rt["active"][:rt_o["n_active"]], rt_o["active"])

    h_in = gu.h_in_from_gpu(lay, res)
    c = orc.layer_chain(lay, h_in=h_in, rows=rows)
    f = orc.layer_f64(lay, h_in=h_in, rows=rows)
    mask = np.zeros((R, k), bool)
    mask[rt_o["pair_row"], rt_o["pair_slot"]] = True
    if rows is not None:
        keep = np.zeros(R, bool)
        keep[list(rows)] = True
        mask &= keep[:, None]
    gud = gu.per_pair(res, "gu_dbg", lay)
    hd = gu.per_pair(res, "h_dbg", lay)
    # accumulators: bit-exact
    assert gu.bits_equal(gud[:, :, 0][mask], c["g"][mask]), "g differs from the fp32-chain oracle"
    assert gu.bits_equal(gud[:, :, 1][mask], c["u"][mask]), "u differs from the fp32-chain oracle"
    # h before quantisation: within the float64 bound
    assert orc.within_tol(hd[mask], f["h"][mask], f["mh"][mask]).all()
    # quantised h: the oracle's quantiser on the device's fp32 h gives the device's codes
    for p in range(n):
        r, j = int(rt_o["pair_row"][p]), int(rt_o["pair_slot"][p])
        if not mask[r, j]:
            continue
        q, s = orc.quantize_act(kind, res["h_dbg"][p])
        if kind == synth.ACT_E4M3:
            assert np.array_equal(res["h"][p], q) and np.array_equal(res["h_scale"][p], s), (r, j)
        else:
            assert gu.bf16_equal(res["h"][p].view(np.uint16), q), (r, j)
    # down: bit-exact against the chain oracle fed with the device's h; within the bound
    dm = res["out"][mask]
    assert gu.bits_equal(dm, c["d"][mask]), "d differs from the fp32-chain oracle"
    assert orc.within_tol(dm, f["d"][mask], f["md"][mask]).all()
    # combine: bit-exact, and within the bound (+ half a bf16 ulp for the final rounding)
    rows_all = range(R) if rows is None else rows
    for r in rows_all:
        if not mask[r].all():
            continue  # rows with a left-out slot combine unwritten entries
        assert gu.bits_equal(res["y_f32"][r], c["y_f32"][r])
        assert gu.bf16_equal(res["y"][r].view(np.uint16), c["y_bf16"][r])
        yb = orc.bf16_to_f32(res["y"][r].view(np.uint16)).astype(np.float64)
        half_ulp = np.abs(f["y"][r]) * 2.0 ** -8
        assert orc.within_tol(yb, f["y"][r], f["my"][r], extra=half_ulp).all()
    return c, f


def test_route_matches_oracle(orc):
    rng = np.random.default_rng(0)
    for trial in range(30):
        E = int(rng.choice([8, 64, 256, 1024]))
        k = int(rng.integers(1, min(E, 9)))
        R = int(rng.choice([0, 1, 3, 16, 100, 4096 if trial % 10 == 0 else 50]))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(R)]).astype(np.int32) if R else np.zeros((0, k), np.int32)
        if trial % 3 == 0 and R:
            ids[rng.integers(0, R), rng.integers(0, k)] = rng.choice([-1, E, 5 * E])
            if k > 1:
                r = rng.integers(0, R)
                ids[r, -1] = ids[r, 0]
        d = tfx.dims(64, 32, E, k)
        rt = tfx.alloc_route(R, E, k, gu.DEV)
        st = torch.zeros(1, dtype=torch.int32, device=gu.DEV)
        idd = torch.from_numpy(ids.copy()).to(gu.DEV) if R else torch.zeros(1, dtype=torch.int32, device=gu.DEV)
        tfx.tfx_xp_route(d, R, idd, rt, st)
        torch.cuda.synchronize()
        ref = orc.route(ids.reshape(R, k), E)
        n = int(ref["offs"][-1])
        assert int(st.item()) == ref["status"]
        assert np.array_equal(rt["offs"].cpu().numpy(), ref["offs"])
        assert np.array_equal(rt["pair_row"].cpu().numpy()[:n], ref["pair_row"])
        assert np.array_equal(rt["pair_slot"].cpu().numpy()[:n], ref["pair_slot"])
        assert int(rt["n_active"].item()) == ref["n_active"]
        assert np.array_equal(rt["active"].cpu().numpy()[:ref["n_active"]], ref["active"])


@pytest.mark.parametrize("shape", [(700, 3, 64), (1537, 8, 256), (1537, 8, 1024), (4096, 8, 256), (3001, 1, 8)],
                         ids=["3-ctas", "13-ctas", "13-ctas-unstaged", "32-ctas", "ragged"])
def test_route_in_several_ctas_matches_oracle(orc, shape):
    # launches above 2,048 pairs split the scatter over CTAs (each counts every pair itself)
    R, k, E = shape
    rng = np.random.default_rng(R + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(R)]).astype(np.int32)
    for _ in range(7):  # out-of-range ids and duplicates, spread over the blocks
        ids[rng.integers(0, R), rng.integers(0, k)] = rng.choice([-1, E, 5 * E])
        if k > 1:
            r = rng.integers(0, R)
            ids[r, -1] = ids[r, 0]
    d = tfx.dims(64, 32, E, k)
    rt = tfx.alloc_route(R, E, k, gu.DEV)
    st = torch.zeros(1, dtype=torch.int32, device=gu.DEV)
    tfx.tfx_xp_route(d, R, torch.from_numpy(ids).to(gu.DEV), rt, st)
    torch.cuda.synchronize()
    ref = orc.route(ids, E)
    n = int(ref["offs"][-1])
    assert int(st.item()) == ref["status"]
    assert np.array_equal(rt["offs"].cpu().numpy(), ref["offs"])
    assert np.array_equal(rt["pair_row"].cpu().numpy()[:n], ref["pair_row"])
    assert np.array_equal(rt["pair_slot"].cpu().numpy()[:n], ref["pair_slot"])
    assert int(rt["n_active"].item()) == ref["n_active"]
    assert np.array_equal(rt["active"].cpu().numpy()[:ref["n_active"]], ref["active"])


def test_pack_layout(orc):
    """The packed stage layout, rebuilt here on the host from the canonical arrays."""
    lay = small_layer(synth.ACT_E4M3, H=1088, I=96, E=3, k=2, R=1, seed=4)
    H, I, E = lay["H"], lay["I"], lay["E"]
    d = tfx.dims(H, I, E, 2)
    packed = gu.pack(d, gu.device_weights_from_numpy(lay)).cpu().numpy()
    S, Sd = (H + 511) // 512, (I + 511) // 512
    STAGE = 64 * 272
    exp = []
    for e in range(E):
        for u in range(I // 32):
            for s in range(S):
                codes = np.zeros((64, 256), np.uint8)
                sc = np.zeros((64, 16), np.uint8)
                for rho in range(64):
                    wc, ws = (lay["wg"], lay["sg"]) if rho < 32 else (lay["wu"], lay["su"])
                    n = 32 * u + rho % 32
                    cb = wc[e, n, 256 * s:256 * s + 256]
                    codes[rho, :cb.size] = cb
                    sb = ws[e, n, 16 * s:16 * s + 16]
                    sc[rho, :sb.size] = sb
                exp.append(codes.ravel())
                exp.append(sc.ravel())
    for e in range(E):
        for u in range(H // 64):
            for s in range(Sd):
                codes = np.zeros((64, 256), np.uint8)
                sc = np.zeros((64, 16), np.uint8)
                for rho in range(64):
                    m = 64 * u + rho
                    cb = lay["wd"][e, m, 256 * s:256 * s + 256]
                    codes[rho, :cb.size] = cb
                    sb = lay["sd"][e, m, 16 * s:16 * s + 16]
                    sc[rho, :sb.size] = sb
                exp.append(codes.ravel())
                exp.append(sc.ravel())
    exp = np.concatenate(exp)
    assert exp.size == packed.size == E * ((I // 32) * S + (H // 64) * Sd) * STAGE
    assert np.array_equal(exp, packed)


@pytest.mark.parametrize("kind", [synth.ACT_BF16, synth.ACT_E4M3], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("shape", [dict(H=256, I=128, E=8, k=2, R=4), dict(H=1088, I=96, E=16, k=4, R=7),
                                   dict(H=2048, I=544, E=6, k=3, R=13)], ids=["tiny", "ragged", "stages"])
def test_layer_parity(orc, kind, shape):
    lay = small_layer(kind, seed=7, **shape)
    d = tfx.dims(lay["H"], lay["I"], lay["E"], lay["ids"].shape[1])
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    res = gu.run_layer(lay, packed)
    check_layer(orc, lay, res)


@pytest.mark.parametrize("kind", [synth.ACT_BF16, synth.ACT_E4M3], ids=["bf16", "e4m3"])
def test_extreme_values_parity(orc, kind):
    """Large and tiny activations: bf16 groups that need the exact fallback (exponent spread
    beyond the f16 window, values near the ends of the range), scale codes at 0 and 254."""
    lay = small_layer(kind, H=512, I=64, E=4, k=2, R=4, seed=3)
    rng = np.random.default_rng(3)
    if kind == synth.ACT_BF16:
        z = rng.standard_normal((4, 512)).astype(np.float32)
        z[0, :32] *= np.float32(2.0 ** 40)         # one group far from the rest, still one window
        z[0, 40] = np.float32(2.0 ** -60)          # spread > 32 binades inside a group: fallback
        z[1, 64:96] *= np.float32(2.0 ** -120)     # tiny group (subnormal products)
        z[2, 100] = np.float32(2.0 ** 100)         # very large value
        z[3, 200] = np.float32(2.0 ** -130)        # bf16 subnormal
        lay["x"], _ = synth.activations(z, kind)
    else:
        lay["sx"][0, 0] = 0
        lay["sx"][1, 1] = 254
        lay["sx"][2, 2] = 200
        lay["sg"][:, :, 0] = 0
        lay["su"][:, :, 1] = 254
    d = tfx.dims(lay["H"], lay["I"], lay["E"], 2)
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    res = gu.run_layer(lay, packed)
    # finite checks only where the float64 reference is finite
    R, k = lay["ids"].shape
    h_in = gu.h_in_from_gpu(lay, res)
    c = orc.layer_chain(lay, h_in=h_in)
    gud = gu.per_pair(res, "gu_dbg", lay)
    assert gu.bits_equal(gud[:, :, 0], c["g"]) and gu.bits_equal(gud[:, :, 1], c["u"])
    assert gu.bits_equal(res["out"], c["d"])
    assert gu.bits_equal(res["y_f32"], c["y_f32"])


def test_invalid_ids_are_reported_and_left_out(orc):
    lay = small_layer(synth.ACT_E4M3, H=256, I=64, E=8, k=3, R=5, seed=5)
    lay["ids"][1, 2] = 8        # out of range
    lay["ids"][3, 1] = lay["ids"][3, 0]  # duplicate
    d = tfx.dims(lay["H"], lay["I"], lay["E"], 3)
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    res = gu.run_layer(lay, packed, canary=0xA5)
    assert res["status"] & tfx.ST_RANGE and res["status"] & tfx.ST_DUP
    canary = np.full(4, 0xA5, np.uint8).view(np.float32)[0]
    assert np.all(res["out"][1, 2].view(np.uint32) == canary.view(np.uint32))
    assert np.all(res["out"][3, 1].view(np.uint32) == canary.view(np.uint32))
    check_layer(orc, lay, res, rows=[0, 2, 4])


def test_zero_rows():
    d = tfx.dims(256, 128, 8, 2)
    buf = tfx.alloc_layer(0, 256, 128, 8, 2, synth.ACT_E4M3, gu.DEV)
    packed = torch.zeros(tfx.tfx_xp_packed_bytes(d), dtype=torch.uint8, device=gu.DEV)
    x = torch.zeros(16, dtype=torch.uint8, device=gu.DEV)
    ids = torch.zeros(1, dtype=torch.int32, device=gu.DEV)
    w = torch.zeros(1, dtype=torch.float32, device=gu.DEV)
    tfx.layer_rows(d, 0, synth.ACT_E4M3, packed, x, x, ids, w, buf)
    torch.cuda.synchronize()
    assert int(buf["status"].item()) == 0 and int(buf["route"]["n_active"].item()) == 0


def test_bounded_wait_reports_timeout():
    st = torch.zeros(1, dtype=torch.int32, device=gu.DEV)
    tfx.tfx_selftest_wait_timeout(st, 2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert int(st.item()) == tfx.ST_TIMEOUT
    # the context is still usable afterwards
    assert float(torch.ones(4, device=gu.DEV).sum().item()) == 4.0
