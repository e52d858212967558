"""The C-ABI library builds for sm_103a, loads, exports every function include/tfx_moe.h
declares, and rejects bad arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tfx_moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(tfx_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from moe_routed_expert_major_gb300 import build, tfx
    build.build()
    return tfx.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tfx_xp_route", "tfx_xp_upc_rows", "tfx_xp_down_rows", "tfx_xp_combine", "tfx_xp_pack",
              "tfx_xp_packed_bytes", "tfx_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_packed_size(lib):
    from moe_routed_expert_major_gb300 import tfx
    # 256 experts x (22,020,096 code bytes + 1,376,256 scale bytes): no padding at these widths
    assert tfx.tfx_xp_packed_bytes(tfx.dims(7168, 2048, 256, 8)) == 256 * 23396352
    assert tfx.tfx_xp_packed_bytes(tfx.dims(100, 2048, 256, 8)) == 0   # H not a multiple of 64


def test_invalid_arguments_are_rejected_before_launch(lib):
    from moe_routed_expert_major_gb300 import tfx
    d = tfx.dims(7168, 2048, 256, 8)
    bad = tfx.dims(7168, 2048, 0, 8)
    st = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    rt = tfx.Route(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16))
    L = lib
    assert L.tfx_xp_route(bad, 1, st, st, st, st, st, st, st, None) == -1
    assert L.tfx_xp_route(d, -1, st, st, st, st, st, st, st, None) == -1
    assert L.tfx_xp_route(d, 1, None, st, st, st, st, st, st, None) == -1
    # upc: null packed, misaligned x, bad kind, bad max_pass
    assert L.tfx_xp_upc_rows(d, 1, 0, None, st, st, ctypes.byref(rt), st, st, None, None, st, None, None) == -1
    assert L.tfx_xp_upc_rows(d, 1, 0, st, ctypes.c_void_p(17), st, ctypes.byref(rt), st, st, None, None, st, None, None) == -1
    assert L.tfx_xp_upc_rows(d, 1, 7, st, st, st, ctypes.byref(rt), st, st, None, None, st, None, None) == -1
    o = tfx.opts_struct(max_pass=3)
    assert L.tfx_xp_upc_rows(d, 1, 0, st, st, st, ctypes.byref(rt), st, st, None, None, st, ctypes.byref(o), None) == -1
    o = tfx.opts_struct(max_pass=8)
    assert L.tfx_xp_down_rows(d, 1, 0, st, st, st, ctypes.byref(rt), st, st, ctypes.byref(o), None) == -1
    assert L.tfx_xp_down_rows(d, 1, 0, st, st, st, None, st, st, None, None) == -1
    assert L.tfx_xp_combine(tfx.dims(100, 2048, 256, 8), 1, st, st, st, None, None) == -1
    assert L.tfx_xp_combine(d, 1, None, st, st, None, None) == -1
    assert L.tfx_xp_pack(bad, st, st, st, st, st, st, st, None) == -1
    assert L.tfx_selftest_wait_timeout(None, 1000, None) == -1
    assert L.tfx_strerror(-2) == b"unsupported shape for these kernels"


def test_chunk_entries_reject_before_launch(lib):
    """The chunk path covers E4M3 activations with H and I multiples of 512 only."""
    from moe_routed_expert_major_gb300 import tfx
    d = tfx.dims(7168, 2048, 256, 8)
    st = ctypes.c_void_p(64)  # aligned for every argument
    rt = tfx.Route(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16))
    L = lib
    big = 1 << 40
    up = lambda dd, kind, x=st, xs=st, r=ctypes.byref(rt), ws=ctypes.c_void_p(256), wsb=big: L.tfx_xp_upc_chunk(
        dd, 4, kind, st, x, xs, r, st, st, None, None, ws, wsb, st, None, None)
    assert up(d, 1) == -2                         # bf16 activations
    assert up(tfx.dims(7168 + 256, 2048, 256, 8), 0) == -2  # H not a multiple of 512
    assert up(tfx.dims(7168, 2048 + 128, 256, 8), 0) == -2  # I not a multiple of 512
    assert up(tfx.dims(7168, 2048, 0, 8), 0) == -1
    assert up(d, 0, x=ctypes.c_void_p(24)) == -1  # x not 16-byte aligned
    assert up(d, 0, xs=ctypes.c_void_p(72)) == -1  # x_scale not 16-byte aligned
    assert up(d, 0, r=None) == -1
    assert L.tfx_xp_upc_chunk(d, 4, 0, ctypes.c_void_p(16), st, st, ctypes.byref(rt), st, st, None, None,
                              ctypes.c_void_p(256), big, st, None, None) == -1  # packed not 32-byte aligned
    assert up(d, 0, ws=None) == -1                       # no workspace
    assert up(d, 0, wsb=L.tfx_xp_upc_chunk_ws_bytes(d, 4) - 1) == -1  # workspace too small
    assert L.tfx_xp_upc_chunk_ws_bytes(d, 4096) == 32768 * 7168 + 32768 * 224
    assert L.tfx_xp_down_chunk(d, 4, 0, st, st, st, ctypes.byref(rt), None, st, None, None) == -1
    assert L.tfx_xp_down_chunk(d, 4, 1, st, st, st, ctypes.byref(rt), st, st, None, None) == -2
    assert L.tfx_xp_down_chunk(d, 0, 0, st, st, st, ctypes.byref(rt), st, st, None, None) == 0  # R = 0: no-op


def test_router_entries_reject_before_launch(lib):
    """Both routers check their sizes, mode and pointers before any launch; R = 0 is a no-op."""
    L = lib
    p = ctypes.c_void_p(64)  # never dereferenced: validation fails first
    assert L.tfx_xp_router(1, 0, 1, p, 0, -1, p, p, None) == -1          # no logits
    assert L.tfx_xp_router(1, 1025, 8, p, 0, -1, p, p, None) == -1       # more than 1,024 logits
    assert L.tfx_xp_router(1, 256, 33, p, 0, -1, p, p, None) == -1       # top_k above 32
    assert L.tfx_xp_router(1, 4, 5, p, 0, -1, p, p, None) == -1          # top_k above n_logits
    assert L.tfx_xp_router(1, 256, 8, p, 2, -1, p, p, None) == -1        # unknown mode
    assert L.tfx_xp_router(1, 256, 8, p, 0, -2, p, p, None) == -1        # bad shared expert
    assert L.tfx_xp_router(1, 256, 8, None, 0, -1, p, p, None) == -1     # null logits
    assert L.tfx_xp_router(0, 256, 8, None, 0, -1, None, None, None) == 0
    g = lambda rows=1, n=256, k=8, lg=p, ng=8, kg=4, sc=1.0, sh=-1, ids=p, w=p: L.tfx_xp_router_grouped(
        rows, n, k, lg, None, ng, kg, sc, sh, ids, w, None)
    assert g(ng=0) == -1 and g(ng=33) == -1            # group count out of range
    assert g(n=250) == -1                              # groups do not divide the experts
    assert g(n=8, ng=8, kg=1, k=1) == -1               # groups of one expert
    assert g(kg=0) == -1 and g(kg=9) == -1             # kept groups out of range
    assert g(n=64, ng=8, kg=1, k=9) == -1              # top_k above the kept experts
    assert g(sc=float("nan")) == -1                    # NaN scale
    assert g(sh=-2) == -1 and g(lg=None) == -1 and g(w=None) == -1
    assert g(rows=0, lg=None, ids=None, w=None) == 0
