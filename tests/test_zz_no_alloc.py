"""tfx_xp_moe_rows_noalloc: the one-launch layer for callers that cannot allocate device
memory (a host runtime that owns every allocation, or a path where an allocation would
synchronise or fail). It keeps its counters in a buffer built into the library instead of
caller scratch; here two calls in a row must give the same results, bit for bit, as the
entry point that takes caller scratch, and a launch too large for the built-in buffer must be
refused before anything runs. This file is collected last on purpose."""
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


def _run_noalloc(lay, packed):
    R, k = lay["ids"].shape
    d = tfx.dims(lay["H"], lay["I"], lay["E"], k)
    xd, xs, ids, w = gu.to_dev_inputs(lay)
    buf = tfx.alloc_layer(R, lay["H"], lay["I"], lay["E"], k, lay["kind"], gu.DEV, debug=True)
    tfx.tfx_xp_moe_rows_noalloc(d, R, lay["kind"], packed, xd, xs, ids, w, buf["route"], buf["h"], buf["h_scale"],
                                buf["out"], buf["y"], buf["status"], buf["y_f32"])
    torch.cuda.synchronize()
    res = {n: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for n, v in buf.items() if n != "route"}
    res["route"] = {n: v.cpu().numpy() for n, v in buf["route"].items()}
    res["status"] = int(buf["status"].item())
    return res


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16], ids=["e4m3", "bf16"])
@pytest.mark.parametrize("shape", [dict(H=256, I=128, E=8, k=2, R=4), dict(H=1088, I=96, E=16, k=4, R=7)],
                         ids=["tiny", "ragged"])
def test_noalloc_matches_caller_scratch_twice(kind, shape):
    cfg = synth.workload("tiny", kind=kind, seed=23, **{n: v for n, v in shape.items() if n != "R"})
    lay = synth.make_layer_numpy(cfg, R=shape["R"])
    d = tfx.dims(lay["H"], lay["I"], lay["E"], lay["ids"].shape[1])
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    ref, _ = gu.run_layer_fused(lay, packed)
    assert ref["status"] == 0
    for _ in range(2):  # the built-in buffer keeps the last call's contents: the second call must not mind
        got = _run_noalloc(lay, packed)
        assert got["status"] == 0
        gu.assert_same_layer(got, ref, lay)


def test_noalloc_full_width_decode_twice():
    cfg = synth.workload("decode")
    lay, dw = gu.full_layer(cfg)
    d = tfx.dims(cfg["H"], cfg["I"], cfg["E"], cfg["k"])
    packed = gu.pack(d, dw)
    ref, _ = gu.run_layer_fused(lay, packed)
    for _ in range(2):
        got = _run_noalloc(lay, packed)
        assert got["status"] == 0
        gu.assert_same_layer(got, ref, lay)


def test_noalloc_refusals_run_without_a_device():
    """The refusal cases (a launch beyond the built-in buffer, bad arguments) in a child
    process that sees no CUDA device, so that no check that ever went missing could launch
    on their made-up addresses."""
    from test_abi import run_without_device
    run_without_device("noalloc")
