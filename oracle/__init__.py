"""CPU oracle for routed-expert MoE over MXFP4 weights -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package. The CUDA library never calls it; the two share no code.

The arithmetic lives in ``tfx_oracle.c`` (plain C, one output at a time). This module only
marshals numpy arrays, loops over (row, slot) pairs and runs pairs on several host threads
(ctypes drops the GIL during each call; every output is computed by one thread alone, so the
thread count never changes a bit).

Definitions follow "dsv41 metal: decode experts decode an expert's weights once for all of
its rows" (TensorFold PR #2983): "What this changes" and the rows kernels' commit message.
Every function with no independent pin says so in its docstring; the pins are in
``tests/test_oracle_*.py``.
"""
import ctypes
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

ACT_E4M3 = 0
ACT_BF16 = 1
ST_RANGE = 1
ST_DUP = 2

_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            sig = {
                "tfxo_e2m1_value": (ctypes.c_double, [_I]),
                "tfxo_e4m3_value": (ctypes.c_double, [_I]),
                "tfxo_ue8m0_value": (ctypes.c_double, [_I]),
                "tfxo_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "tfxo_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "tfxo_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
                "tfxo_e4m3_encode": (_I, [ctypes.c_double]),
                "tfxo_quant_e4m3_f32": (None, [_I, _P, _P, _P]),
                "tfxo_quant_e4m3_f64": (None, [_I, _P, _P, _P]),
                "tfxo_round_bf16": (None, [_I, _P, _P]),
                "tfxo_round_bf16_f64": (None, [_I, _P, _P]),
                "tfxo_route": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
                "tfxo_chain_dot": (ctypes.c_float, [_I, _P, _P, _P, _P]),
                "tfxo_f64_dot": (ctypes.c_double, [_I, _P, _P, _P, _P]),
                "tfxo_gateup_chain": (None, [_I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P]),
                "tfxo_gateup_f64": (None, [_I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P]),
                "tfxo_silu_mul_f32": (None, [_I, _P, _P, _P]),
                "tfxo_silu_mul_f64": (None, [_I, _P, _P, _P, _P, _P, _P]),
                "tfxo_down_chain": (None, [_I, _I, _P, _P, _I, _P, _P, _P, _P]),
                "tfxo_down_f64": (None, [_I, _I, _P, _P, _I, _P, _P, _P, _P, _P]),
                "tfxo_combine_chain": (None, [_I, _I, _P, _P, _P, _P]),
                "tfxo_combine_f64": (None, [_I, _I, _P, _P, _P, _P, _P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads():
    return max(1, os.cpu_count() or 1)


# ------------------------------------------------------------------ element formats

def e2m1_value(code):
    return lib().tfxo_e2m1_value(int(code))


def e4m3_value(code):
    return lib().tfxo_e4m3_value(int(code))


def ue8m0_value(code):
    return lib().tfxo_ue8m0_value(int(code))


def e4m3_encode(v):
    """Nearest E4M3 code (ties to even, saturating at 448) of each float64 in ``v``."""
    v = np.asarray(v, dtype=np.float64).ravel()
    return np.array([lib().tfxo_e4m3_encode(float(t)) for t in v], dtype=np.uint8)


def f32_to_bf16(a):
    a = np.ascontiguousarray(a, dtype=np.float32).ravel()
    out = np.empty(a.shape, dtype=np.uint16)
    lib().tfxo_round_bf16(a.size, _p(a), _p(out))
    return out


def f64_to_bf16(a):
    """Each float64 rounded once, to nearest even, straight to bf16 bits (no binary32 step)."""
    a = np.ascontiguousarray(a, dtype=np.float64).ravel()
    out = np.empty(a.shape, dtype=np.uint16)
    lib().tfxo_round_bf16_f64(a.size, _p(a), _p(out))
    return out


def bf16_to_f32(b):
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def quant_e4m3(h):
    """Block quantiser of a fp32 vector (length a multiple of 32) -> (codes u8, scales u8)."""
    h = np.ascontiguousarray(h, dtype=np.float32).ravel()
    assert h.size % 32 == 0
    codes = np.empty(h.size, np.uint8)
    scales = np.empty(h.size // 32, np.uint8)
    lib().tfxo_quant_e4m3_f32(h.size, _p(h), _p(codes), _p(scales))
    return codes, scales


def quant_e4m3_f64(h):
    h = np.ascontiguousarray(h, dtype=np.float64).ravel()
    assert h.size % 32 == 0
    codes = np.empty(h.size, np.uint8)
    scales = np.empty(h.size // 32, np.uint8)
    lib().tfxo_quant_e4m3_f64(h.size, _p(h), _p(codes), _p(scales))
    return codes, scales


# ------------------------------------------------------------------ routing

def route(ids, E):
    """Expert-major row lists from top-k ids [R, k] (see tfx_oracle.c, routing)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    R, k = ids.shape
    offs = np.zeros(E + 1, np.int32)
    P = R * k
    pair_row = np.full(max(P, 1), -1, np.int32)
    pair_slot = np.full(max(P, 1), -1, np.int32)
    active = np.full(max(min(P, E), 1), -1, np.int32)
    n_active = np.zeros(1, np.int32)
    st = lib().tfxo_route(_p(ids), R, k, E, _p(offs), _p(pair_row), _p(pair_slot), _p(active), _p(n_active))
    n = int(offs[E])
    na = int(n_active[0])
    return dict(status=int(st), offs=offs, pair_row=pair_row[:n].copy(), pair_slot=pair_slot[:n].copy(),
                active=active[:na].copy(), n_active=na)


def router(logits, k, mode=0, shared=-1):
    """Routing ids and weights from router logits [R, n] (float64 arithmetic).

    The pages take the routing as given; this follows the library's own routing convention
    (the conventions of the synthetic inputs, which the rows kernels consume): the k largest
    logits of a row, equal values going to the lower expert id, in descending order; NaN ranks
    below every number (taken only when a row has fewer than k numbers), -0 equals +0.
    mode 0: w_j = exp(l_j - l_0) / sum over the selected slots; mode 1: sigmoid scores
    1 / (1 + exp(-l_j)) normalised to sum 1. shared >= 0 appends that expert id to every row
    with weight 1. Returns (ids int32 [R, k (+1)], w float64 [R, k (+1)])."""
    L = np.asarray(logits, np.float64)
    R, n = L.shape
    nan = np.isnan(L)
    v = np.where(nan, 0.0, L)
    idx = np.arange(n)
    ids = np.zeros((R, k), np.int32)
    w = np.zeros((R, k), np.float64)
    for r in range(R):
        order = np.lexsort((idx, -v[r], nan[r]))[:k]  # numbers first, then larger, then lower id
        sel = L[r, order]
        with np.errstate(over="ignore", invalid="ignore"):  # -inf or NaN logits give 0, inf or NaN
            t = np.exp(sel - sel[0]) if mode == 0 else 1.0 / (1.0 + np.exp(-sel))
        ids[r] = order
        with np.errstate(invalid="ignore"):
            w[r] = t / t.sum()
    if shared >= 0:
        ids = np.concatenate([ids, np.full((R, 1), shared, np.int32)], axis=1)
        w = np.concatenate([w, np.ones((R, 1))], axis=1)
    return ids, w


# fp32 constants of sigmoid32: 1/ln 2; ln 2 split after Cody and Waite into a 16-bit head
# (n * head is exact for |n| < 128) and the rest; the Taylor coefficients 1/j! of exp.
_F32 = np.float32
_LOG2E = _F32(1.4426950408889634)
_LN2_HI = _F32(0.693145751953125)
_LN2_LO = _F32(0.6931471805599453 - 0.693145751953125)
_INV_FACT = [_F32(1.0 / f) for f in (1, 1, 2, 6, 24, 120, 720, 5040)]


def sigmoid32(l):
    """The grouped router's sigmoid, every step one IEEE fp32 operation rounded to nearest.

    t = exp(y) for y = max(-|l|, -86): n = rint(y / ln 2), r = (y - n*LN2_HI) - n*LN2_LO,
    exp(r) by its degree-7 Taylor polynomial in Horner form (multiply, then add), times 2^n;
    then 1 / (1 + t) for l >= 0 and t / (1 + t) for l < 0. NaN stays NaN. Logits below -86
    are taken as -86 (their sigmoid is below 5e-38), so no step meets a subnormal."""
    l = np.asarray(l, np.float32)
    nan = np.isnan(l)
    lz = np.where(nan, _F32(0.0), l)
    y = np.maximum(-np.abs(lz), _F32(-86.0))
    n = np.rint(y * _LOG2E)
    r = (y - n * _LN2_HI) - n * _LN2_LO
    p = np.full_like(r, _INV_FACT[7])
    for c in _INV_FACT[6::-1]:
        p = p * r + c
    two_n = ((n.astype(np.int32) + 127) << 23).astype(np.int32).view(np.float32)
    t = p * two_n
    d = _F32(1.0) + t
    s = np.where(lz >= 0, _F32(1.0) / d, t / d)
    return np.where(nan, l, s).astype(np.float32)


def _rank(v):
    """Indices of v ordered by value, larger first, equal values by lower index, NaN last
    (-0 equals +0)."""
    v = np.asarray(v, np.float64)
    nan = np.isnan(v)
    return np.lexsort((np.arange(v.size), -np.where(nan, 0.0, v), nan))


def router_grouped(logits, k, n_group, topk_group, bias=None, scale=1.0, shared=-1):
    """Group-limited sigmoid routing (DeepSeek-V3 style), all arithmetic in fp32.

    Per row: s = sigmoid32(l); choice scores c = s + bias (fp32 add; bias omitted: c = s). The
    n experts form n_group contiguous groups of n / n_group; a group's score is the sum, in
    fp32, of its two best choice scores (best first). The topk_group best groups are kept
    (equal scores: lower group first); the k best experts of the kept groups by c are the ids,
    in that order (equal scores: lower id first; NaN ranks below every number). Weights:
    w_j = (s_j / S) * scale, S = s_0 + s_1 + ... summed in slot order in fp32 from +0. The
    bias steers the choice only, never the weights. shared >= 0 appends that expert with
    weight 1. Returns (ids int32 [R, k (+1)], w float32 [R, k (+1)])."""
    L = np.asarray(logits, np.float32)
    R, n = L.shape
    gs = n // n_group
    s = sigmoid32(L)
    c = s + np.asarray(bias, np.float32)[None, :] if bias is not None else s
    ids = np.zeros((R, k), np.int32)
    w = np.zeros((R, k), np.float32)
    for r in range(R):
        G = np.zeros(n_group, np.float32)
        for g in range(n_group):
            grp = c[r, g * gs:(g + 1) * gs]
            top = _rank(grp)[:2]
            G[g] = _F32(grp[top[0]]) + _F32(grp[top[1]])
        kept = _rank(G)[:topk_group]
        allowed = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in sorted(kept)])
        sel = allowed[_rank(c[r, allowed])[:k]]
        ids[r] = sel
        ssum = _F32(0.0)
        for e in sel:
            ssum = _F32(ssum + s[r, e])
        with np.errstate(invalid="ignore"):
            w[r] = (s[r, sel] / ssum) * _F32(scale)
    if shared >= 0:
        ids = np.concatenate([ids, np.full((R, 1), shared, np.int32)], axis=1)
        w = np.concatenate([w, np.ones((R, 1), np.float32)], axis=1)
    return ids, w


# ------------------------------------------------------------------ one output

def chain_dot(wc, ws, xc, xs):
    """fp32 chain of one output. wc: codes [K/2] u8, ws: scales [K/32] u8, xc: unscaled
    activation values fp32 [K], xs: activation group scales fp32 [K/32]."""
    wc = np.ascontiguousarray(wc, np.uint8)
    ws = np.ascontiguousarray(ws, np.uint8)
    xc = np.ascontiguousarray(xc, np.float32)
    xs = np.ascontiguousarray(xs, np.float32)
    return lib().tfxo_chain_dot(xc.size, _p(wc), _p(ws), _p(xc), _p(xs))


def f64_dot(wc, ws, xh):
    wc = np.ascontiguousarray(wc, np.uint8)
    ws = np.ascontiguousarray(ws, np.uint8)
    xh = np.ascontiguousarray(xh, np.float64)
    m = ctypes.c_double(0.0)
    v = lib().tfxo_f64_dot(xh.size, _p(wc), _p(ws), _p(xh), ctypes.byref(m))
    return v, m.value


# ------------------------------------------------------------------ one (expert, row) pair

def _act_row(layer, r):
    if layer["kind"] == ACT_E4M3:
        return layer["x"][r], layer["sx"][r]
    return layer["x"][r], None


def gateup_chain(layer, e, r):
    H, I = layer["H"], layer["I"]
    x, sx = _act_row(layer, r)
    g = np.empty(I, np.float32)
    u = np.empty(I, np.float32)
    buf = np.empty(H + H // 32, np.float32)
    lib().tfxo_gateup_chain(H, I, _p(layer["wg"][e]), _p(layer["sg"][e]), _p(layer["wu"][e]), _p(layer["su"][e]),
                            layer["kind"], _p(x), _p(sx), _p(buf), _p(g), _p(u))
    return g, u


def gateup_f64(layer, e, r):
    H, I = layer["H"], layer["I"]
    x, sx = _act_row(layer, r)
    g = np.empty(I)
    u = np.empty(I)
    mg = np.empty(I)
    mu = np.empty(I)
    buf = np.empty(H)
    lib().tfxo_gateup_f64(H, I, _p(layer["wg"][e]), _p(layer["sg"][e]), _p(layer["wu"][e]), _p(layer["su"][e]),
                          layer["kind"], _p(x), _p(sx), _p(buf), _p(g), _p(u), _p(mg), _p(mu))
    return g, u, mg, mu


def silu_mul(g, u):
    g = np.ascontiguousarray(g, np.float32)
    u = np.ascontiguousarray(u, np.float32)
    h = np.empty_like(g)
    lib().tfxo_silu_mul_f32(g.size, _p(g), _p(u), _p(h))
    return h


def silu_mul_f64(g, u, mg, mu):
    g, u, mg, mu = (np.ascontiguousarray(a, np.float64) for a in (g, u, mg, mu))
    h = np.empty_like(g)
    mh = np.empty_like(g)
    lib().tfxo_silu_mul_f64(g.size, _p(g), _p(u), _p(mg), _p(mu), _p(h), _p(mh))
    return h, mh


def quantize_act(kind, h):
    """The launch's activation format for h: E4M3 codes + scales, or bf16 bits (scales None)."""
    if kind == ACT_E4M3:
        return quant_e4m3(h)
    return f32_to_bf16(h), None


def down_chain(layer, e, hq, hs):
    H, I = layer["H"], layer["I"]
    hq = np.ascontiguousarray(hq)
    hs = None if hs is None else np.ascontiguousarray(hs, np.uint8)
    d = np.empty(H, np.float32)
    buf = np.empty(I + I // 32, np.float32)
    lib().tfxo_down_chain(H, I, _p(layer["wd"][e]), _p(layer["sd"][e]), layer["kind"], _p(hq), _p(hs), _p(buf), _p(d))
    return d


def down_f64(layer, e, hq, hs):
    H, I = layer["H"], layer["I"]
    hq = np.ascontiguousarray(hq)
    hs = None if hs is None else np.ascontiguousarray(hs, np.uint8)
    d = np.empty(H)
    md = np.empty(H)
    buf = np.empty(I)
    lib().tfxo_down_f64(H, I, _p(layer["wd"][e]), _p(layer["sd"][e]), layer["kind"], _p(hq), _p(hs), _p(buf), _p(d), _p(md))
    return d, md


def combine_chain(d, w):
    """One row: d [k, H] fp32, w [k] fp32 -> (y bf16 bits [H], y fp32 [H])."""
    d = np.ascontiguousarray(d, np.float32)
    w = np.ascontiguousarray(w, np.float32)
    k, H = d.shape
    yb = np.empty(H, np.uint16)
    yf = np.empty(H, np.float32)
    lib().tfxo_combine_chain(k, H, _p(d), _p(w), _p(yb), _p(yf))
    return yb, yf


def combine_f64(d, md, w):
    d = np.ascontiguousarray(d, np.float64)
    md = np.ascontiguousarray(md, np.float64)
    w = np.ascontiguousarray(w, np.float32)
    k, H = d.shape
    y = np.empty(H)
    my = np.empty(H)
    lib().tfxo_combine_f64(k, H, _p(d), _p(md), _p(w), _p(y), _p(my))
    return y, my


# ------------------------------------------------------------------ whole layer

def _pairs(layer):
    ids = layer["ids"]
    rt = route(ids, layer["E"])
    pairs = [(int(rt["pair_row"][p]), int(rt["pair_slot"][p]), int(ids[rt["pair_row"][p], rt["pair_slot"][p]]))
             for p in range(len(rt["pair_row"]))]
    return rt, pairs


def _map(fn, items, threads):
    threads = threads or default_threads()
    if threads <= 1 or len(items) <= 1:
        return [fn(it) for it in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


def layer_chain(layer, h_in=None, threads=None, rows=None):
    """fp32-chain evaluation of a whole layer.

    ``layer`` holds H, I, E, k, kind, weights in canonical layout (wg, sg, wu, su, wd, sd),
    activations (x and, for E4M3, sx), ids [R, k] and w [R, k].
    ``h_in`` optionally replaces the quantised activation fed to the down projection: a dict
    {(r, j): (codes_or_bf16, scales_or_None)}, so a test can feed a device's own h.
    ``rows`` restricts the work to those rows (outputs of other rows stay zero).
    Returns per-(row, slot) arrays g, u, h [R, k, I] fp32, hq/hs (quantised h), d [R, k, H]
    fp32, and y_bf16 [R, H], y_f32 [R, H].
    """
    R, k = layer["ids"].shape
    H, I, kind = layer["H"], layer["I"], layer["kind"]
    rt, pairs = _pairs(layer)
    if rows is not None:
        rows = set(int(r) for r in rows)
        pairs = [p for p in pairs if p[0] in rows]
    g = np.zeros((R, k, I), np.float32)
    u = np.zeros((R, k, I), np.float32)
    h = np.zeros((R, k, I), np.float32)
    hq = np.zeros((R, k, I), np.uint8 if kind == ACT_E4M3 else np.uint16)
    hs = np.zeros((R, k, I // 32), np.uint8)
    d = np.zeros((R, k, H), np.float32)

    def one(pr):
        r, j, e = pr
        gg, uu = gateup_chain(layer, e, r)
        hh = silu_mul(gg, uu)
        q, s = quantize_act(kind, hh)
        if h_in is not None:
            q, s = h_in[(r, j)]
        dd = down_chain(layer, e, q, s)
        return pr, gg, uu, hh, q, s, dd

    for (r, j, e), gg, uu, hh, q, s, dd in _map(one, pairs, threads):
        g[r, j], u[r, j], h[r, j], hq[r, j], d[r, j] = gg, uu, hh, q, dd
        if s is not None:
            hs[r, j] = s
    yb = np.zeros((R, H), np.uint16)
    yf = np.zeros((R, H), np.float32)
    for r in range(R):
        if rows is not None and r not in rows:
            continue
        yb[r], yf[r] = combine_chain(d[r], layer["w"][r])
    return dict(route=rt, g=g, u=u, h=h, hq=hq, hs=hs, d=d, y_bf16=yb, y_f32=yf)


def layer_f64(layer, h_in=None, threads=None, rows=None):
    """float64 evaluation with masses. ``h_in`` as in :func:`layer_chain`; without it the
    down consumes the float64 h quantised by the same rule. Returns g, u, h, d, y and their
    masses mg, mu, mh, md, my."""
    R, k = layer["ids"].shape
    H, I, kind = layer["H"], layer["I"], layer["kind"]
    rt, pairs = _pairs(layer)
    if rows is not None:
        rows = set(int(r) for r in rows)
        pairs = [p for p in pairs if p[0] in rows]
    out = {n: np.zeros((R, k, I)) for n in ("g", "u", "h", "mg", "mu", "mh")}
    out["d"] = np.zeros((R, k, H))
    out["md"] = np.zeros((R, k, H))

    def one(pr):
        r, j, e = pr
        gg, uu, mg, mu = gateup_f64(layer, e, r)
        hh, mh = silu_mul_f64(gg, uu, mg, mu)
        if h_in is not None:
            q, s = h_in[(r, j)]
        elif kind == ACT_E4M3:
            q, s = quant_e4m3_f64(hh)
        else:
            q, s = f64_to_bf16(hh), None  # h rounded once, from float64, to nearest even
        dd, md = down_f64(layer, e, q, s)
        return pr, gg, uu, hh, mg, mu, mh, dd, md

    for (r, j, e), gg, uu, hh, mg, mu, mh, dd, md in _map(one, pairs, threads):
        out["g"][r, j], out["u"][r, j], out["h"][r, j] = gg, uu, hh
        out["mg"][r, j], out["mu"][r, j], out["mh"][r, j] = mg, mu, mh
        out["d"][r, j], out["md"][r, j] = dd, md
    out["y"] = np.zeros((R, H))
    out["my"] = np.zeros((R, H))
    for r in range(R):
        if rows is not None and r not in rows:
            continue
        out["y"][r], out["my"][r] = combine_f64(out["d"][r], out["md"][r], layer["w"][r])
    out["route"] = rt
    return out


def within_tol(got, ref, mass, rel=1e-3, abs_=1e-6, extra=0.0):
    """The tolerance |got - ref| <= rel * mass + abs + extra, elementwise (NaN must match NaN)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both_nan = np.isnan(got) & np.isnan(ref)
    err = np.abs(got - ref)
    ok = (err <= rel * np.asarray(mass) + abs_ + extra) | both_nan
    return ok
