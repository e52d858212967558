"""Thin ctypes binding of libtfx_moe.so (the C ABI in include/tfx_moe.h).

Argument marshalling only: every function takes torch CUDA tensors, passes their device
pointers and the current CUDA stream to the C entry point of the same name, and raises on
a negative return code. No arithmetic of the method happens here, and there is no fallback:
if the library is missing, loading fails.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libtfx_moe.so")

ACT_E4M3 = 0
ACT_BF16 = 1
ST_RANGE = 1
ST_DUP = 2
ST_TIMEOUT = 4
ST_SHAPE = 8


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32)]


class Route(ctypes.Structure):
    _fields_ = [("offs", ctypes.c_void_p), ("pair_row", ctypes.c_void_p), ("pair_slot", ctypes.c_void_p),
                ("active", ctypes.c_void_p), ("n_active", ctypes.c_void_p)]


class RowsOpts(ctypes.Structure):
    _fields_ = [("max_pass", ctypes.c_int32), ("tier_mode", ctypes.c_int32), ("timeout_ns", ctypes.c_int64)]


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32


def load():
    """Load the in-tree shared library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libtfx_moe.so is not built (run moe_routed_expert_major_gb300/build.py or "
                               "__graft_entry__.build()); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "tfx_xp_packed_bytes": (ctypes.c_size_t, [Dims]),
            "tfx_xp_pack": (ctypes.c_int, [Dims, _P, _P, _P, _P, _P, _P, _P, _P]),
            "tfx_xp_route": (ctypes.c_int, [Dims, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
            "tfx_xp_upc_rows": (ctypes.c_int, [Dims, _I32, _I32, _P, _P, _P, ctypes.POINTER(Route), _P, _P, _P, _P, _P,
                                               ctypes.POINTER(RowsOpts), _P]),
            "tfx_xp_down_rows": (ctypes.c_int, [Dims, _I32, _I32, _P, _P, _P, ctypes.POINTER(Route), _P, _P,
                                                ctypes.POINTER(RowsOpts), _P]),
            "tfx_xp_upc_chunk_ws_bytes": (ctypes.c_size_t, [Dims, _I32]),
            "tfx_xp_upc_chunk": (ctypes.c_int, [Dims, _I32, _I32, _P, _P, _P, ctypes.POINTER(Route), _P, _P, _P, _P, _P,
                                                ctypes.c_size_t, _P, ctypes.POINTER(RowsOpts), _P]),
            "tfx_xp_down_chunk": (ctypes.c_int, [Dims, _I32, _I32, _P, _P, _P, ctypes.POINTER(Route), _P, _P,
                                                ctypes.POINTER(RowsOpts), _P]),
            "tfx_xp_combine": (ctypes.c_int, [Dims, _I32, _P, _P, _P, _P, _P]),
            "tfx_xp_moe_rows_scratch_bytes": (ctypes.c_size_t, [Dims, _I32]),
            "tfx_xp_moe_rows": (ctypes.c_int, [Dims, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                               _P, _P, _P, _P, _P, _P, ctypes.POINTER(RowsOpts), _P]),
            "tfx_xp_moe_rows_noalloc": (ctypes.c_int, [Dims, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                       _P, _P, _P, _P, _P, ctypes.POINTER(RowsOpts), _P]),
            "tfx_xp_moe_rows_host_ws_bytes": (ctypes.c_size_t, [Dims, _I32, _I32]),
            "tfx_xp_moe_rows_host_layout": (ctypes.c_int, [Dims, _I32, _I32, ctypes.POINTER(ctypes.c_size_t),
                                                           ctypes.POINTER(ctypes.c_size_t)]),
            "tfx_xp_moe_rows_host": (ctypes.c_int, [Dims, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                    ctypes.c_size_t, ctypes.POINTER(RowsOpts), _P]),
            "tfx_xp_router": (ctypes.c_int, [_I32, _I32, _I32, _P, _I32, _I32, _P, _P, _P]),
            "tfx_xp_router_grouped": (ctypes.c_int, [_I32, _I32, _I32, _P, _P, _I32, _I32, ctypes.c_float, _I32,
                                                     _P, _P, _P]),
            "tfx_strerror": (ctypes.c_char_p, [ctypes.c_int]),
            "tfx_version": (ctypes.c_int, []),
            "tfx_selftest_wait_timeout": (ctypes.c_int, [_P, ctypes.c_int64, _P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tfx: tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tfx: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _hptr(t):
    """Host tensor -> pointer (pinned memory keeps the copies asynchronous)."""
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("tfx: this argument is a host buffer")
    if not t.is_contiguous():
        raise ValueError("tfx: tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("%s failed: %s (%d)" % (what, load().tfx_strerror(rc).decode(), rc))


def dims(H, I, E, k):
    return Dims(H, I, E, k)


def route_struct(rt):
    return Route(*(ctypes.c_void_p(rt[n].data_ptr()) for n in ("offs", "pair_row", "pair_slot", "active", "n_active")))


def opts_struct(max_pass=0, tier_mode=0, timeout_ns=0):
    return RowsOpts(max_pass, tier_mode, timeout_ns)


# ------------------------------------------------------------------ entry points

def tfx_xp_packed_bytes(d):
    return int(load().tfx_xp_packed_bytes(d))


def tfx_xp_pack(d, w, packed):
    _check(load().tfx_xp_pack(d, _ptr(w["wg"]), _ptr(w["sg"]), _ptr(w["wu"]), _ptr(w["su"]), _ptr(w["wd"]),
                              _ptr(w["sd"]), _ptr(packed), _stream()), "tfx_xp_pack")


def tfx_xp_route(d, rows, ids, rt, status):
    _check(load().tfx_xp_route(d, rows, _ptr(ids), _ptr(rt["offs"]), _ptr(rt["pair_row"]), _ptr(rt["pair_slot"]),
                               _ptr(rt["active"]), _ptr(rt["n_active"]), _ptr(status), _stream()), "tfx_xp_route")


def tfx_xp_upc_rows(d, rows, kind, packed, x, x_scale, rt, h, h_scale, status, gu_dbg=None, h_dbg=None, opts=None):
    r = route_struct(rt)
    o = ctypes.byref(opts) if opts is not None else None
    _check(load().tfx_xp_upc_rows(d, rows, kind, _ptr(packed), _ptr(x), _ptr(x_scale), ctypes.byref(r), _ptr(h),
                                  _ptr(h_scale), _ptr(gu_dbg), _ptr(h_dbg), _ptr(status), o, _stream()),
           "tfx_xp_upc_rows")


def tfx_xp_down_rows(d, rows, kind, packed, h, h_scale, rt, out, status, opts=None):
    r = route_struct(rt)
    o = ctypes.byref(opts) if opts is not None else None
    _check(load().tfx_xp_down_rows(d, rows, kind, _ptr(packed), _ptr(h), _ptr(h_scale), ctypes.byref(r), _ptr(out),
                                   _ptr(status), o, _stream()), "tfx_xp_down_rows")


def tfx_xp_upc_chunk_ws_bytes(d, rows):
    return int(load().tfx_xp_upc_chunk_ws_bytes(d, rows))


def tfx_xp_upc_chunk(d, rows, kind, packed, x, x_scale, rt, h, h_scale, ws, status, gu_dbg=None, h_dbg=None,
                     opts=None):
    r = route_struct(rt)
    o = ctypes.byref(opts) if opts is not None else None
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().tfx_xp_upc_chunk(d, rows, kind, _ptr(packed), _ptr(x), _ptr(x_scale), ctypes.byref(r), _ptr(h),
                                   _ptr(h_scale), _ptr(gu_dbg), _ptr(h_dbg), _ptr(ws), nbytes, _ptr(status), o,
                                   _stream()),
           "tfx_xp_upc_chunk")


def tfx_xp_down_chunk(d, rows, kind, packed, h, h_scale, rt, out, status, opts=None):
    r = route_struct(rt)
    o = ctypes.byref(opts) if opts is not None else None
    _check(load().tfx_xp_down_chunk(d, rows, kind, _ptr(packed), _ptr(h), _ptr(h_scale), ctypes.byref(r), _ptr(out),
                                    _ptr(status), o, _stream()), "tfx_xp_down_chunk")


def tfx_xp_combine(d, rows, out, topk_w, y, y_f32=None):
    _check(load().tfx_xp_combine(d, rows, _ptr(out), _ptr(topk_w), _ptr(y), _ptr(y_f32), _stream()),
           "tfx_xp_combine")


def tfx_xp_moe_rows_scratch_bytes(d, rows):
    return int(load().tfx_xp_moe_rows_scratch_bytes(d, rows))


def tfx_xp_moe_rows(d, rows, kind, packed, x, x_scale, ids, topk_w, rt, h, h_scale, out, y, scratch, status,
                    y_f32=None, opts=None, gu_dbg=None, h_dbg=None):
    o = ctypes.byref(opts) if opts is not None else None
    _check(load().tfx_xp_moe_rows(d, rows, kind, _ptr(packed), _ptr(x), _ptr(x_scale), _ptr(ids), _ptr(topk_w),
                                  _ptr(rt["offs"]), _ptr(rt["pair_row"]), _ptr(rt["pair_slot"]), _ptr(rt["active"]),
                                  _ptr(rt["n_active"]), _ptr(h), _ptr(h_scale), _ptr(out), _ptr(y), _ptr(y_f32),
                                  _ptr(gu_dbg), _ptr(h_dbg), _ptr(scratch), _ptr(status), o, _stream()),
           "tfx_xp_moe_rows")


def tfx_xp_moe_rows_noalloc(d, rows, kind, packed, x, x_scale, ids, topk_w, rt, h, h_scale, out, y, status,
                            y_f32=None, opts=None):
    """tfx_xp_moe_rows with the library's built-in counter buffer instead of caller scratch."""
    o = ctypes.byref(opts) if opts is not None else None
    _check(load().tfx_xp_moe_rows_noalloc(d, rows, kind, _ptr(packed), _ptr(x), _ptr(x_scale), _ptr(ids),
                                          _ptr(topk_w), _ptr(rt["offs"]), _ptr(rt["pair_row"]), _ptr(rt["pair_slot"]),
                                          _ptr(rt["active"]), _ptr(rt["n_active"]), _ptr(h), _ptr(h_scale), _ptr(out),
                                          _ptr(y), _ptr(y_f32), _ptr(status), o, _stream()),
           "tfx_xp_moe_rows_noalloc")


def tfx_xp_moe_rows_host_ws_bytes(d, rows, kind):
    return int(load().tfx_xp_moe_rows_host_ws_bytes(d, rows, kind))


def tfx_xp_moe_rows_host_layout(d, rows, kind):
    """(byte offsets of x, x_scale, ids and topk_w in one host input block, the block's size)."""
    off = (ctypes.c_size_t * 4)()
    n = ctypes.c_size_t()
    _check(load().tfx_xp_moe_rows_host_layout(d, rows, kind, off, ctypes.byref(n)), "tfx_xp_moe_rows_host_layout")
    return [int(v) for v in off], int(n.value)


def tfx_xp_moe_rows_host(d, rows, kind, packed, x_host, x_scale_host, ids_host, topk_w_host, y_host, status, ws,
                         status_host=None, opts=None):
    """The one-launch layer from host buffers: copy in, the layer, copy y (and the status) out, all
    queued on the current stream. packed, status and ws live on the device; the rest on the host."""
    o = ctypes.byref(opts) if opts is not None else None
    _check(load().tfx_xp_moe_rows_host(d, rows, kind, _ptr(packed), _hptr(x_host), _hptr(x_scale_host),
                                       _hptr(ids_host), _hptr(topk_w_host), _hptr(y_host), _ptr(status),
                                       _hptr(status_host), _ptr(ws), ws.numel() * ws.element_size(), o, _stream()),
           "tfx_xp_moe_rows_host")


ROUTER_SOFTMAX = 0
ROUTER_SIGMOID = 1


def tfx_xp_router(logits, top_k, ids, topk_w, mode=ROUTER_SOFTMAX, shared_expert=-1):
    """ids [R][k (+1)] int32 and topk_w [R][k (+1)] fp32 from logits [R][n] fp32 (device)."""
    R, n = int(logits.shape[0]), int(logits.shape[1])
    _check(load().tfx_xp_router(R, n, int(top_k), _ptr(logits), int(mode), int(shared_expert), _ptr(ids),
                                _ptr(topk_w), _stream()), "tfx_xp_router")


def tfx_xp_router_grouped(logits, top_k, n_group, topk_group, ids, topk_w, bias=None, scale=1.0, shared_expert=-1):
    """Group-limited sigmoid routing: ids [R][k (+1)] int32 and topk_w [R][k (+1)] fp32 from
    logits [R][n] fp32 and an optional bias [n] fp32 (device)."""
    R, n = int(logits.shape[0]), int(logits.shape[1])
    _check(load().tfx_xp_router_grouped(R, n, int(top_k), _ptr(logits), _ptr(bias),
                                        int(n_group), int(topk_group), float(scale), int(shared_expert), _ptr(ids),
                                        _ptr(topk_w), _stream()), "tfx_xp_router_grouped")


def tfx_selftest_wait_timeout(status, timeout_ns):
    _check(load().tfx_selftest_wait_timeout(_ptr(status), int(timeout_ns), _stream()), "tfx_selftest_wait_timeout")


# ------------------------------------------------------------------ buffers (allocation only)

def alloc_route(R, E, k, device):
    P = max(R * k, 1)
    i32 = dict(dtype=torch.int32, device=device)
    return dict(offs=torch.zeros(E + 1, **i32), pair_row=torch.zeros(P, **i32), pair_slot=torch.zeros(P, **i32),
                active=torch.zeros(max(min(R * k, E), 1), **i32), n_active=torch.zeros(1, **i32))


def alloc_layer(R, H, I, E, k, kind, device, debug=False, chunk=False):
    """Output and intermediate buffers of one layer launch of R rows (chunk=True adds the gate/up
    chunk path's workspace)."""
    P = max(R * k, 1)
    b = dict(route=alloc_route(R, E, k, device), status=torch.zeros(1, dtype=torch.int32, device=device))
    if kind == ACT_E4M3:
        b["h"] = torch.empty(P, I, dtype=torch.uint8, device=device)
        b["h_scale"] = torch.empty(P, I // 32, dtype=torch.uint8, device=device)
    else:
        b["h"] = torch.empty(P, I, dtype=torch.int16, device=device)
        b["h_scale"] = None
    b["out"] = torch.empty(max(R, 1), k, H, dtype=torch.float32, device=device)
    b["y"] = torch.empty(max(R, 1), H, dtype=torch.int16, device=device)
    nsc = tfx_xp_moe_rows_scratch_bytes(Dims(H, I, E, k), max(R, 1)) // 4
    b["scratch"] = torch.zeros(max(nsc, 1), dtype=torch.int32, device=device)
    b["chunk_ws"] = None
    if chunk:
        b["chunk_ws"] = torch.empty(max(tfx_xp_upc_chunk_ws_bytes(Dims(H, I, E, k), R), 1), dtype=torch.uint8,
                                    device=device)
    if debug:
        b["gu_dbg"] = torch.empty(P, 2, I, dtype=torch.float32, device=device)
        b["h_dbg"] = torch.empty(P, I, dtype=torch.float32, device=device)
        b["y_f32"] = torch.empty(max(R, 1), H, dtype=torch.float32, device=device)
    else:
        b["gu_dbg"] = b["h_dbg"] = b["y_f32"] = None
    return b


def layer_fused(d, R, kind, packed, x, x_scale, ids, w, buf, opts=None):
    """One MoE layer of R rows in a single launch (tfx_xp_moe_rows)."""
    tfx_xp_moe_rows(d, R, kind, packed, x, x_scale, ids, w, buf["route"], buf["h"], buf["h_scale"], buf["out"],
                    buf["y"], buf["scratch"], buf["status"], buf["y_f32"], opts, buf["gu_dbg"], buf["h_dbg"])


def layer_chunk(d, R, kind, packed, x, x_scale, ids, w, buf, opts=None):
    """One MoE layer of R rows on the chunk path: route -> gate/up chunk -> down chunk ->
    combine, four launches on the current stream."""
    tfx_xp_route(d, R, ids, buf["route"], buf["status"])
    tfx_xp_upc_chunk(d, R, kind, packed, x, x_scale, buf["route"], buf["h"], buf["h_scale"], buf["chunk_ws"],
                     buf["status"], buf["gu_dbg"], buf["h_dbg"], opts)
    tfx_xp_down_chunk(d, R, kind, packed, buf["h"], buf["h_scale"], buf["route"], buf["out"], buf["status"], opts)
    tfx_xp_combine(d, R, buf["out"], w, buf["y"], buf["y_f32"])


def layer_rows(d, R, kind, packed, x, x_scale, ids, w, buf, opts_upc=None, opts_down=None):
    """One MoE layer of R rows: route -> gate/up -> down -> combine, four launches on the
    current stream (no host synchronisation)."""
    tfx_xp_route(d, R, ids, buf["route"], buf["status"])
    tfx_xp_upc_rows(d, R, kind, packed, x, x_scale, buf["route"], buf["h"], buf["h_scale"], buf["status"],
                    buf["gu_dbg"], buf["h_dbg"], opts_upc)
    tfx_xp_down_rows(d, R, kind, packed, buf["h"], buf["h_scale"], buf["route"], buf["out"], buf["status"], opts_down)
    tfx_xp_combine(d, R, buf["out"], w, buf["y"], buf["y_f32"])
