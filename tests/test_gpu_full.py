"""Parity at the full DeepSeek-class widths (H 7168, I 2048, E 256, top-8), in the launch
configuration the benchmark times: every output of the 1-row decode layer, and sampled rows
of the shared-routing (R 16), routed-apart bf16 (R 4, NaN/Inf planted) and 4,096-row layers,
checked bit for bit against the fp32-chain oracle and within the float64 bound."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import gpu_util as gu  # noqa: E402
from moe_routed_expert_major_gb300 import tfx  # noqa: E402
from test_gpu_parity import check_layer  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_routed_expert_major_gb300 import build
    build.build()
    tfx.load()


def _packed_layer(cfg, R=None):
    lay, dw = gu.full_layer(cfg, R=R)
    d = tfx.dims(cfg["H"], cfg["I"], cfg["E"], cfg["k"])
    packed = gu.pack(d, dw)
    return lay, packed


def test_decode_one_row_every_output(orc):
    cfg = synth.workload("decode")
    lay, packed = _packed_layer(cfg)
    res = gu.run_layer(lay, packed)
    assert res["status"] == 0
    check_layer(orc, lay, res)


@pytest.mark.parametrize("R", [2, 5, 16])
def test_shared_routing_sampled_rows(orc, R):
    cfg = synth.workload("shared")
    lay, packed = _packed_layer(cfg, R=R)
    res = gu.run_layer(lay, packed)
    assert res["status"] == 0
    assert int(res["route"]["n_active"][0]) == 8
    check_layer(orc, lay, res, rows=sorted({0, R // 2, R - 1}))
    # row 0 alone gives the same bits
    one = dict(lay)
    one["x"], one["sx"], one["ids"], one["w"] = lay["x"][:1], lay["sx"][:1], lay["ids"][:1], lay["w"][:1]
    alone = gu.run_layer(one, packed)
    assert np.array_equal(res["y"][0].view(np.uint16), alone["y"][0].view(np.uint16))
    assert np.array_equal(res["out"][0].view(np.uint32), alone["out"][0].view(np.uint32))


def test_apart_bf16_with_nonfinite_row(orc):
    cfg = synth.workload("apart")
    lay, packed = _packed_layer(cfg, R=4)
    clean = dict(lay)
    clean["x"] = lay["x"].copy()
    synth.plant_nonfinite(lay, 1, seed=3)
    res = gu.run_layer(lay, packed)
    assert res["status"] == 0
    check_layer(orc, lay, res, rows=[0, 2, 3])
    y1 = orc.bf16_to_f32(res["y"][1].view(np.uint16))
    assert np.isnan(y1).any()
    cres = gu.run_layer(clean, packed)
    for r in (0, 2, 3):
        assert np.array_equal(res["y"][r].view(np.uint16), cres["y"][r].view(np.uint16))


def test_chunk_rows_sampled(orc):
    cfg = synth.workload("chunk")
    lay, packed = _packed_layer(cfg)
    res = gu.run_layer(lay, packed)
    assert res["status"] == 0
    assert int(res["route"]["offs"][-1]) == 4096 * 8
    check_layer(orc, lay, res, rows=[0, 1777, 4095])
