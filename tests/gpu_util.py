"""Helpers for the GPU tests: put a layer on the device, pack it, run it through the C ABI,
and bring the results back as numpy. The oracle side reads the same inputs from host copies.
"""
import numpy as np
import torch

import synth
from moe_routed_expert_major_gb300 import tfx

DEV = "cuda:0"


class LazyExperts:
    """Host view of device weights [E, ...]: experts are copied back on first use."""

    def __init__(self, t):
        self.t = t
        self.cache = {}
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = np.ascontiguousarray(self.t[e].cpu().numpy())
        return self.cache[e]


def device_weights_from_numpy(lay):
    return {n: torch.from_numpy(np.ascontiguousarray(lay[n])).to(DEV) for n in ("wg", "sg", "wu", "su", "wd", "sd")}


def pack(d, w):
    packed = torch.empty(tfx.tfx_xp_packed_bytes(d), dtype=torch.uint8, device=DEV)
    tfx.tfx_xp_pack(d, w, packed)
    return packed


def full_layer(cfg, R=None, seed=None):
    """Full-size layer: weights drawn on the device, inputs on the host. Returns (lay, dw)
    where lay is the oracle's dict (weights as lazy host views)."""
    seed = cfg["seed"] if seed is None else seed
    dw = synth.weights_torch(cfg["E"], cfg["H"], cfg["I"], seed, DEV)
    lay = dict(H=cfg["H"], I=cfg["I"], E=cfg["E"], k=cfg["k"], kind=cfg["kind"])
    for n, t in dw.items():
        lay[n] = LazyExperts(t)
    lay.update(synth.make_inputs(cfg, R=R, seed=seed))
    return lay, dw


def to_dev_inputs(lay):
    x = lay["x"]
    if lay["kind"] == synth.ACT_BF16:
        xd = torch.from_numpy(x.view(np.int16).copy()).to(DEV)
        xs = None
    else:
        xd = torch.from_numpy(x.copy()).to(DEV)
        xs = torch.from_numpy(lay["sx"].copy()).to(DEV)
    ids = torch.from_numpy(lay["ids"].astype(np.int32).copy()).to(DEV)
    w = torch.from_numpy(lay["w"].astype(np.float32).copy()).to(DEV)
    return xd, xs, ids, w


def run_layer(lay, packed, debug=True, opts_upc=None, opts_down=None, canary=None):
    """Run route + gate/up + down + combine on the device; return numpy results."""
    R, k = lay["ids"].shape
    d = tfx.dims(lay["H"], lay["I"], lay["E"], k)
    xd, xs, ids, w = to_dev_inputs(lay)
    buf = tfx.alloc_layer(R, lay["H"], lay["I"], lay["E"], k, lay["kind"], DEV, debug=debug)
    if canary is not None:
        for n in ("h", "h_scale", "out", "y", "gu_dbg", "h_dbg", "y_f32"):
            if buf.get(n) is not None:
                buf[n].view(torch.uint8).fill_(canary)
    tfx.layer_rows(d, R, lay["kind"], packed, xd, xs, ids, w, buf, opts_upc, opts_down)
    torch.cuda.synchronize()
    res = {n: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for n, v in buf.items() if n != "route"}
    res["route"] = {n: v.cpu().numpy() for n, v in buf["route"].items()}
    res["status"] = int(buf["status"].item())
    return res


def run_layer_chunk(lay, packed, debug=True, canary=None):
    """Route + gate/up + down on the chunk path (tensor cores) + combine; numpy results."""
    R, k = lay["ids"].shape
    d = tfx.dims(lay["H"], lay["I"], lay["E"], k)
    xd, xs, ids, w = to_dev_inputs(lay)
    buf = tfx.alloc_layer(R, lay["H"], lay["I"], lay["E"], k, lay["kind"], DEV, debug=debug, chunk=True)
    if canary is not None:
        for n in ("h", "h_scale", "out", "y", "gu_dbg", "h_dbg", "y_f32"):
            if buf.get(n) is not None:
                buf[n].view(torch.uint8).fill_(canary)
    tfx.layer_chunk(d, R, lay["kind"], packed, xd, xs, ids, w, buf)
    torch.cuda.synchronize()
    res = {n: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for n, v in buf.items()
           if n not in ("route", "chunk_ws")}
    res["route"] = {n: v.cpu().numpy() for n, v in buf["route"].items()}
    res["status"] = int(buf["status"].item())
    return res


def h_in_from_gpu(lay, res):
    """The device's quantised h, keyed by (row, slot), for the oracle's down stage."""
    rt = res["route"]
    n = int(rt["offs"][-1])
    out = {}
    for p in range(n):
        r, j = int(rt["pair_row"][p]), int(rt["pair_slot"][p])
        if lay["kind"] == synth.ACT_E4M3:
            out[(r, j)] = (res["h"][p].copy(), res["h_scale"][p].copy())
        else:
            out[(r, j)] = (res["h"][p].view(np.uint16).copy(), None)
    return out


def per_pair(res, name, lay):
    """Reorder a per-pair device array [P, ...] into [R, k, ...] (zeros where unrouted)."""
    R, k = lay["ids"].shape
    rt = res["route"]
    a = res[name]
    out = np.zeros((R, k) + a.shape[1:], a.dtype)
    for p in range(int(rt["offs"][-1])):
        out[rt["pair_row"][p], rt["pair_slot"][p]] = a[p]
    return out


def bits_equal(a, b):
    """Bitwise equality of float arrays, with every NaN equal to every NaN."""
    a = np.asarray(a)
    b = np.asarray(b)
    if a.shape != b.shape:
        return False
    fa = a.astype(np.float64)
    fb = b.astype(np.float64)
    nan = np.isnan(fa) & np.isnan(fb)
    ua = a.view(np.uint32 if a.dtype == np.float32 else np.uint16 if a.dtype.itemsize == 2 else np.uint8)
    ub = b.view(ua.dtype)
    return bool(np.all((ua == ub) | nan))


def bf16_equal(a, b):
    """Bitwise equality of bf16 bit patterns, with every NaN equal to every NaN."""
    fa = (np.asarray(a).view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    fb = (np.asarray(b).view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return bits_equal(fa, fb)


def run_layer_fused(lay, packed, opts=None, canary=None, scratch=None):
    """The whole layer in one launch (tfx_xp_moe_rows); returns numpy results and the scratch."""
    R, k = lay["ids"].shape
    d = tfx.dims(lay["H"], lay["I"], lay["E"], k)
    xd, xs, ids, w = to_dev_inputs(lay)
    buf = tfx.alloc_layer(R, lay["H"], lay["I"], lay["E"], k, lay["kind"], DEV, debug=True)
    if scratch is not None:
        buf["scratch"] = scratch
    if canary is not None:
        for n in ("h", "h_scale", "out", "y", "y_f32"):
            if buf.get(n) is not None:
                buf[n].view(torch.uint8).fill_(canary)
    tfx.layer_fused(d, R, lay["kind"], packed, xd, xs, ids, w, buf, opts)
    torch.cuda.synchronize()
    res = {n: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for n, v in buf.items() if n != "route"}
    res["route"] = {n: v.cpu().numpy() for n, v in buf["route"].items()}
    res["status"] = int(buf["status"].item())
    return res, buf["scratch"]


def assert_same_layer(a, b, lay, rows=None):
    """Fused and separate launches: identical row lists, h, d and combine output."""
    R, k = lay["ids"].shape
    n = int(a["route"]["offs"][-1])
    assert np.array_equal(a["route"]["offs"], b["route"]["offs"])
    assert np.array_equal(a["route"]["pair_row"][:n], b["route"]["pair_row"][:n])
    assert np.array_equal(a["route"]["pair_slot"][:n], b["route"]["pair_slot"][:n])
    assert int(a["route"]["n_active"][0]) == int(b["route"]["n_active"][0])
    assert np.array_equal(a["h"][:n].view(np.uint8), b["h"][:n].view(np.uint8))
    if a["h_scale"] is not None:
        assert np.array_equal(a["h_scale"][:n], b["h_scale"][:n])
    routed = set(zip(a["route"]["pair_row"][:n].tolist(), a["route"]["pair_slot"][:n].tolist()))
    rows = range(R) if rows is None else rows
    for r in rows:
        for j in range(k):
            if (r, j) in routed:
                assert np.array_equal(a["out"][r, j].view(np.uint32), b["out"][r, j].view(np.uint32)), (r, j)
        assert np.array_equal(a["y"][r].view(np.uint16), b["y"][r].view(np.uint16)), r
        assert np.array_equal(a["y_f32"][r].view(np.uint32), b["y_f32"][r].view(np.uint32)), r
