"""The router (tfx_xp_router) against the oracle's router: identical ids (ties, signed zeros,
NaN), weights within a few fp32 ulps of float64, the shared-expert slot, and a whole layer
routed on the device with a shared expert against the oracle's layer on its own routing."""
import numpy as np
import pytest

import oracle
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


def run_router(L, k, mode, shared=-1):
    R = L.shape[0]
    s = k + (1 if shared >= 0 else 0)
    ld = torch.from_numpy(np.ascontiguousarray(L, np.float32)).to(gu.DEV)
    ids = torch.full((R, s), -7, dtype=torch.int32, device=gu.DEV)
    w = torch.full((R, s), -7.0, dtype=torch.float32, device=gu.DEV)
    tfx.tfx_xp_router(ld, k, ids, w, mode=mode, shared_expert=shared)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def check(L, k, mode, shared=-1):
    ids, w = run_router(L, k, mode, shared)
    oid, ow = oracle.router(L.astype(np.float32), k, mode, shared)
    assert np.array_equal(ids, oid)
    fin = np.isfinite(ow)
    # fp32: the logit difference, expf (2 ulp), the slot-order sum and the division
    assert np.all(np.abs(w[fin] - ow[fin]) <= 1e-6 * np.abs(ow[fin]) + 1e-30)


@pytest.mark.parametrize("mode", [tfx.ROUTER_SOFTMAX, tfx.ROUTER_SIGMOID], ids=["softmax", "sigmoid"])
@pytest.mark.parametrize("shape", [(256, 256, 8), (37, 1000, 32), (5, 33, 1), (64, 8, 8)],
                         ids=["decode", "wide", "ragged", "all"])
def test_router_matches_the_oracle(mode, shape):
    R, n, k = shape
    L = np.random.default_rng(R * 1000 + n).standard_normal((R, n)).astype(np.float32) * 3
    check(L, k, mode)


def test_router_ties_zeros_nan_and_infinities():
    rng = np.random.default_rng(3)
    L = rng.integers(-2, 3, size=(40, 64)).astype(np.float32)  # many equal values
    L[0, :] = 0.0
    L[1, ::2] = -0.0
    L[2, 5] = np.nan
    L[2, 7] = np.inf
    L[3, :] = np.nan
    L[3, 10:14] = [1.0, -np.inf, 2.0, -0.0]
    L[4, :] = -np.inf
    for mode in (tfx.ROUTER_SOFTMAX, tfx.ROUTER_SIGMOID):
        ids, _ = run_router(L, 8, mode)
        oid, _ = oracle.router(L, 8, mode)
        assert np.array_equal(ids, oid)
    check(L[:3], 8, tfx.ROUTER_SOFTMAX)


def test_router_shared_slot():
    L = np.random.default_rng(4).standard_normal((9, 256)).astype(np.float32)
    check(L, 8, tfx.ROUTER_SOFTMAX, shared=256)
    ids, w = run_router(L, 8, tfx.ROUTER_SOFTMAX, shared=256)
    assert np.all(ids[:, 8] == 256) and np.all(w[:, 8] == 1.0)


@pytest.mark.parametrize("kind", [synth.ACT_E4M3, synth.ACT_BF16], ids=["e4m3", "bf16"])
def test_layer_routed_on_device_with_a_shared_expert(kind):
    # 8 routed experts plus a shared one (expert 8 of the packed weights), top-2 + shared
    cfg = synth.workload("tiny", kind=kind, E=9, seed=23)
    lay = synth.make_layer_numpy(cfg, R=6)
    L = np.random.default_rng(23).standard_normal((6, 8)).astype(np.float32)
    ids, w = run_router(L, 2, tfx.ROUTER_SOFTMAX, shared=8)
    oid, ow = oracle.router(L, 2, 0, shared=8)
    assert np.array_equal(ids, oid)
    d = tfx.dims(lay["H"], lay["I"], lay["E"], 3)
    packed = gu.pack(d, gu.device_weights_from_numpy(lay))
    dev = dict(lay, ids=ids, w=w)
    got = gu.run_layer_fused(dev, packed)[0]
    assert got["status"] == 0
    olay = dict(lay, ids=oid, w=ow)
    h_in = gu.h_in_from_gpu(olay, got)
    c = oracle.layer_chain(dict(olay, w=ow.astype(np.float32)), h_in=h_in)
    f = oracle.layer_f64(olay, h_in=h_in)
    # d does not depend on the routing weights: bit-equal to the chain on the device's h
    n = int(got["route"]["offs"][-1])
    assert n == 6 * 3
    for p in range(n):
        r, j = int(got["route"]["pair_row"][p]), int(got["route"]["pair_slot"][p])
        assert gu.bits_equal(got["out"][r, j], c["d"][r, j])
    # y: the device's and the oracle's weights differ in the last bits: within the bound
    assert oracle.within_tol(got["y_f32"], f["y"], f["my"]).all()


# ------------------------------------------------------------------ group-limited routing

def run_grouped(L, k, ng, kg, bias=None, scale=1.0, shared=-1):
    R = L.shape[0]
    s = k + (1 if shared >= 0 else 0)
    ld = torch.from_numpy(np.ascontiguousarray(L, np.float32)).to(gu.DEV)
    bd = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias, np.float32)).to(gu.DEV)
    ids = torch.full((R, s), -7, dtype=torch.int32, device=gu.DEV)
    w = torch.full((R, s), -7.0, dtype=torch.float32, device=gu.DEV)
    tfx.tfx_xp_router_grouped(ld, k, ng, kg, ids, w, bias=bd, scale=scale, shared_expert=shared)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def check_grouped(L, k, ng, kg, bias=None, scale=1.0, shared=-1):
    ids, w = run_grouped(L, k, ng, kg, bias, scale, shared)
    oid, ow = oracle.router_grouped(L, k, ng, kg, bias, scale, shared)
    # every step is one IEEE fp32 operation on both sides: ids and weight bits are equal (a NaN
    # weight, from NaN logits that had to be taken, is NaN on both sides; its payload may differ)
    assert np.array_equal(ids, oid)
    nan = np.isnan(ow)
    assert np.array_equal(np.isnan(w), nan)
    assert np.array_equal(w[~nan].view(np.uint32), ow[~nan].view(np.uint32))


@pytest.mark.parametrize("shape", [(300, 256, 8, 4, 8), (5, 160, 8, 3, 6), (9, 1024, 32, 4, 32), (17, 64, 32, 32, 8),
                                   (3, 2, 1, 1, 1)],
                         ids=["deepseek", "ragged-groups", "wide", "pairs", "smallest"])
def test_grouped_router_bit_equal_to_the_oracle(shape):
    R, n, ng, kg, k = shape
    rng = np.random.default_rng(R * 7 + n)
    L = (rng.standard_normal((R, n)) * 3).astype(np.float32)
    bias = (rng.standard_normal(n) * 0.1).astype(np.float32)
    check_grouped(L, k, ng, kg, bias, 2.5)
    check_grouped(L, k, ng, kg, None, 1.0)


def test_grouped_router_golden_ties_nan_and_infinities():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "router_grouped.json")) as f:
        for c in json.load(f)["cases"]:
            L = np.array([[float(v) for v in c["logits"]]], np.float32)
            b = None if c["bias"] is None else np.array(c["bias"], np.float32)
            ids, w = run_grouped(L, c["top_k"], c["n_group"], c["topk_group"], b, c["scale"])
            assert ids[0].tolist() == c["ids"], c["name"]
            assert w[0].view(np.uint32).tolist() == [int(v, 16) for v in c["w_bits"]], c["name"]
    rng = np.random.default_rng(31)
    L = (rng.integers(-2, 3, size=(40, 64)) * 0.5).astype(np.float32)  # many equal values
    L[0, :] = 0.0
    L[1, ::2] = -0.0
    L[2, 5] = np.nan
    L[2, 7] = np.inf
    L[3, :] = np.nan
    L[3, 10:14] = [1.0, -np.inf, 2.0, -0.0]
    L[4, :] = -np.inf
    L[5, :] = -200.0
    bias = (rng.integers(-2, 3, size=64) * 0.25).astype(np.float32)
    bias[9] = np.nan
    check_grouped(L, 8, 8, 4, bias, 1.0)
    check_grouped(L, 8, 8, 4, None, 2.5)


def test_grouped_router_shared_slot_and_rejections():
    L = np.random.default_rng(5).standard_normal((9, 256)).astype(np.float32)
    check_grouped(L, 8, 8, 4, None, 2.5, shared=256)
    ids, w = run_grouped(L, 8, 8, 4, None, 2.5, shared=256)
    assert np.all(ids[:, 8] == 256) and np.all(w[:, 8] == 1.0)
    lib = tfx.load()
    x = torch.zeros(4, dtype=torch.float32, device=gu.DEV)
    p = x.data_ptr()
    # groups that do not divide n, groups of one, too many groups kept, k above the kept experts
    assert lib.tfx_xp_router_grouped(1, 10, 2, p, None, 4, 1, 1.0, -1, p, p, None) == -1
    assert lib.tfx_xp_router_grouped(1, 8, 2, p, None, 8, 1, 1.0, -1, p, p, None) == -1
    assert lib.tfx_xp_router_grouped(1, 8, 2, p, None, 4, 5, 1.0, -1, p, p, None) == -1
    assert lib.tfx_xp_router_grouped(1, 8, 5, p, None, 4, 2, 1.0, -1, p, p, None) == -1
    assert lib.tfx_xp_router_grouped(1, 8, 2, None, None, 4, 2, 1.0, -1, p, p, None) == -1
    assert lib.tfx_xp_router_grouped(0, 8, 2, None, None, 4, 2, 1.0, -1, None, None, None) == 0
