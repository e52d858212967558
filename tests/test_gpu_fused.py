"""The one-launch layer (tfx_xp_moe_rows), the launch the benchmark times: against the CPU
oracle at every benchmarked configuration (full DeepSeek-class widths: g, u, d and the combine
bit for bit against the fp32-chain oracle, h within the float64 bound and quantised by the
oracle's rule, every final value within the float64 bound), and against the four separate
launches (identical row lists, h, d and combine output bit for bit) on small and full-width
layers, every pass-size setting and the routing/NaN matrix; its scratch returns to zero after
every call. The host-buffer entry (tfx_xp_moe_rows_host) gives its y bit for bit."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import gpu_util as gu  # noqa: E402
from moe_routed_expert_major_gb300 import tfx  # noqa: E402
from test_gpu_invariance import make_case, ROWS  # noqa: E402
from test_gpu_parity import check_layer  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_routed_expert_major_gb300 import build
    build.build()
    tfx.load()


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16], ids=["e4m3", "bf16"])
@pytest.mark.parametrize("shape", [dict(H=256, I=128, E=8, k=2, R=4), dict(H=1088, I=96, E=16, k=4, R=7),
                                   dict(H=2048, I=544, E=6, k=3, R=13), dict(H=512, I=64, E=40, k=8, R=32)],
                         ids=["tiny", "ragged", "stages", "p256"])
def test_fused_equals_separate(kind, shape):
    cfg = synth.workload("tiny", kind=kind, seed=17, **{n: v for n, v in shape.items() if n != "R"})
    lay = synth.make_layer_numpy(cfg, R=shape["R"])
    d = tfx.dims(lay["H"], lay["I"], lay["E"], lay["ids"].shape[1])
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    sep = gu.run_layer(lay, packed)
    fus, scratch = gu.run_layer_fused(lay, packed)
    assert sep["status"] == 0 and fus["status"] == 0
    gu.assert_same_layer(fus, sep, lay)
    assert int(scratch.abs().sum().item()) == 0
    # a second call on the same scratch gives the same bits
    fus2, _ = gu.run_layer_fused(lay, packed, scratch=scratch)
    gu.assert_same_layer(fus2, sep, lay)
    assert int(scratch.abs().sum().item()) == 0


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16], ids=["e4m3", "bf16"])
def test_fused_matrix_and_pass_sizes(kind):
    from test_gpu_invariance import H, I, E, K
    lay0 = synth.make_layer_numpy(synth.workload("tiny", kind=synth.ACT_E4M3, H=H, I=I, E=E, k=K, seed=99), R=1)
    d = tfx.dims(H, I, E, K)
    packed = gu.pack(d, gu.device_weights_from_numpy(lay0))
    for routing in ("same", "disjoint", "random"):
        for planted in (False, True):
            for R in ROWS:
                lay = make_case(lay0, kind, routing, R, planted, seed=2000 + R)
                sep = gu.run_layer(lay, packed, debug=True)
                fus, _ = gu.run_layer_fused(lay, packed)
                gu.assert_same_layer(fus, sep, lay)
    lay = make_case(lay0, kind, "same", 16, False, seed=5)
    sep = gu.run_layer(lay, packed, debug=True)
    for mp in (1, 2, 3, 4, 5, 6, 7, 8):
        for tm in (0, 1, 2):
            fus, _ = gu.run_layer_fused(lay, packed, opts=tfx.opts_struct(max_pass=mp, tier_mode=tm))
            gu.assert_same_layer(fus, sep, lay)


_TORCH_DT = {np.dtype(np.uint8): torch.uint8, np.dtype(np.int16): torch.int16, np.dtype(np.int32): torch.int32,
             np.dtype(np.float32): torch.float32}


def _host_inputs(lay, d, block, pinned):
    """The layer's x, x_scale, ids and weights in host memory, in one block at the host entry's
    offsets or in four buffers of their own; pinned (the layer reads them in place) or pageable
    (copied to the device: one copy for the block, else one each)."""
    R = lay["ids"].shape[0]
    x = lay["x"].view(np.int16) if lay["kind"] == synth.ACT_BF16 else lay["x"]
    parts = [x, lay["sx"] if lay["kind"] == synth.ACT_E4M3 else None, lay["ids"].astype(np.int32),
             lay["w"].astype(np.float32)]
    parts = [None if a is None else np.ascontiguousarray(a) for a in parts]
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    if not block:
        return [None if a is None else pin(torch.from_numpy(a)) for a in parts]
    off, n = tfx.tfx_xp_moe_rows_host_layout(d, R, lay["kind"])
    blk = pin(torch.zeros(n, dtype=torch.uint8))
    views = []
    for o, a in zip(off, parts):
        if a is None:
            views.append(None)
            continue
        v = blk[o:o + a.nbytes]
        v.copy_(torch.from_numpy(a.reshape(-1).view(np.uint8)))
        views.append(v.view(_TORCH_DT[a.dtype]).view(a.shape))
    return views


@pytest.mark.parametrize("kind,R,block,pinned_in,pinned_y", [
    (synth.ACT_E4M3, 1, True, True, True), (synth.ACT_E4M3, 5, False, False, False),
    (synth.ACT_BF16, 3, True, False, True), (synth.ACT_BF16, 2, False, True, False)],
    ids=["e4m3-1-in-place", "e4m3-5-four-copies", "bf16-3-one-copy", "bf16-2-in-place-y-copied"])
def test_host_entry_equals_device_entry(kind, R, block, pinned_in, pinned_y):
    """tfx_xp_moe_rows_host, one call: inputs read in place from pinned memory or copied from
    pageable memory (one block or four buffers); y stored into pinned memory by the layer or
    copied into pageable memory. Its y equals tfx_xp_moe_rows's bit for bit on the same inputs,
    twice on one workspace."""
    cfg = synth.workload("tiny", kind=kind, seed=23, H=1088, I=96, E=16, k=4)
    lay = synth.make_layer_numpy(cfg, R=R)
    d = tfx.dims(lay["H"], lay["I"], lay["E"], 4)
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    ref, _ = gu.run_layer_fused(lay, packed)
    assert ref["status"] == 0
    xh, xsh, idh, wh = _host_inputs(lay, d, block, pinned_in)
    yh = torch.empty(R, lay["H"], dtype=torch.int16)
    if pinned_y:
        yh = yh.pin_memory()
    sth = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(tfx.tfx_xp_moe_rows_host_ws_bytes(d, R, kind), dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the workspace, its counters back at zero
        yh.fill_(0x5A5A)
        tfx.tfx_xp_moe_rows_host(d, R, kind, packed, xh, xsh, idh, wh, yh, status, ws, status_host=sth)
        torch.cuda.synchronize()
        assert int(sth[0]) == 0
        assert np.array_equal(yh.numpy().view(np.uint16), ref["y"].view(np.uint16))


def test_fused_invalid_ids():
    lay = synth.make_layer_numpy(synth.workload("tiny", kind=synth.ACT_E4M3, H=256, I=64, E=8, k=3, seed=5), R=5)
    lay["ids"][1, 2] = 8
    lay["ids"][3, 1] = lay["ids"][3, 0]
    d = tfx.dims(256, 64, 8, 3)
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    sep = gu.run_layer(lay, packed)
    fus, scratch = gu.run_layer_fused(lay, packed, canary=0x33)
    assert fus["status"] == tfx.ST_RANGE | tfx.ST_DUP
    gu.assert_same_layer(fus, sep, lay, rows=[0, 2, 4])
    # the left-out pairs' outputs are never written
    assert np.all(fus["out"][1, 2].view(np.uint8) == 0x33) and np.all(fus["out"][3, 1].view(np.uint8) == 0x33)
    assert int(scratch.abs().sum().item()) == 0


@pytest.mark.parametrize("name,R", [("decode", 1), ("shared", 16), ("apart", 16)])
def test_fused_full_width(name, R):
    cfg = synth.workload(name)
    lay, dw = gu.full_layer(cfg, R=R)
    d = tfx.dims(cfg["H"], cfg["I"], cfg["E"], cfg["k"])
    packed = gu.pack(d, dw)
    del dw
    sep = gu.run_layer(lay, packed)
    fus, scratch = gu.run_layer_fused(lay, packed)
    assert sep["status"] == 0 and fus["status"] == 0
    gu.assert_same_layer(fus, sep, lay)
    assert int(scratch.abs().sum().item()) == 0


_FULL = {}


def _full_packed(cfg):
    """One full-width weight set per seed (canonical copy for the oracle, packed for the launch)."""
    key = cfg["seed"]
    if key not in _FULL:
        dw = synth.weights_torch(cfg["E"], cfg["H"], cfg["I"], cfg["seed"], gu.DEV)
        d = tfx.dims(cfg["H"], cfg["I"], cfg["E"], cfg["k"])
        _FULL[key] = (dw, gu.pack(d, dw))
    return _FULL[key]


BENCH_CONFIGS = ([("decode", 1, synth.ACT_E4M3)] + [("shared", R, synth.ACT_E4M3) for R in (2, 3, 4, 5, 8, 16)] +
                 [("apart", R, kind) for R in (2, 4, 8, 16) for kind in (synth.ACT_BF16, synth.ACT_E4M3)])


@pytest.mark.parametrize("name,R,kind", BENCH_CONFIGS,
                         ids=["%s-%d-%s" % (n, R, "bf16" if k == synth.ACT_BF16 else "e4m3") for n, R, k in BENCH_CONFIGS])
def test_fused_matches_oracle_at_benchmarked_configs(orc, name, R, kind):
    """The benchmarked launch itself against the oracle: every output of the one-row decode
    layer, and rows 0, R/2 and R-1 of the multi-row layers."""
    cfg = synth.workload(name, kind=kind)
    dw, packed = _full_packed(cfg)
    lay = dict(H=cfg["H"], I=cfg["I"], E=cfg["E"], k=cfg["k"], kind=kind)
    for n, t in dw.items():
        lay[n] = gu.LazyExperts(t)
    lay.update(synth.make_inputs(cfg, R=R))
    res, scratch = gu.run_layer_fused(lay, packed, canary=0x6B)
    assert res["status"] == 0
    rows = None if R == 1 else sorted({0, R // 2, R - 1})
    check_layer(orc, lay, res, rows=rows)
    used = int(res["route"]["offs"][-1])
    assert used == R * cfg["k"]
    assert int(scratch.abs().sum().item()) == 0
