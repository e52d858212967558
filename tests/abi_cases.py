"""Argument-rejection cases of the C ABI, run by tests/test_abi.py and tests/test_zz_no_alloc.py
in a child process that sees no CUDA device (CUDA_VISIBLE_DEVICES empty). The arguments are
made-up addresses that are never dereferenced because validation refuses each call first; in
a process without a device, a check that ever went missing would end in an error code from
the CUDA runtime instead of a launch on those addresses."""
import ctypes
import sys

from moe_routed_expert_major_gb300 import tfx


def rows_and_route(lib):
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
    o = tfx.opts_struct(max_pass=9)
    assert L.tfx_xp_upc_rows(d, 1, 0, st, st, st, ctypes.byref(rt), st, st, None, None, st, ctypes.byref(o), None) == -1
    o = tfx.opts_struct(max_pass=3, tier_mode=3)
    assert L.tfx_xp_upc_rows(d, 1, 0, st, st, st, ctypes.byref(rt), st, st, None, None, st, ctypes.byref(o), None) == -1
    o = tfx.opts_struct(max_pass=8)
    assert L.tfx_xp_down_rows(d, 1, 0, st, st, st, ctypes.byref(rt), st, st, ctypes.byref(o), None) == -1
    assert L.tfx_xp_down_rows(d, 1, 0, st, st, st, None, st, st, None, None) == -1
    assert L.tfx_xp_combine(tfx.dims(100, 2048, 256, 8), 1, st, st, st, None, None) == -1
    assert L.tfx_xp_combine(d, 1, None, st, st, None, None) == -1
    assert L.tfx_xp_pack(bad, st, st, st, st, st, st, st, None) == -1
    assert L.tfx_selftest_wait_timeout(None, 1000, None) == -1
    assert L.tfx_strerror(-2) == b"unsupported shape for these kernels"


def chunk(lib):
    """The chunk path covers E4M3 activations with H and I multiples of 512 only."""
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


def routers(lib):
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



def noalloc(lib):
    """The no-alloc layer refuses a launch beyond its built-in buffer first, then any other bad
    argument, before it touches the buffer."""
    L = lib
    d = tfx.dims(8192, 64, 1024, 2)  # 2 + 1024 + 128 rows * 128 blocks > 16,384 counters
    assert L.tfx_xp_moe_rows_scratch_bytes(d, 128) > 65536
    p = ctypes.c_void_p(256)
    assert L.tfx_xp_moe_rows_noalloc(d, 128, tfx.ACT_E4M3, p, p, p, p, p, p, p, p, p, p, p, p, p, p, None, p, None,
                                     None) == -2
    d = tfx.dims(256, 128, 8, 2)
    assert L.tfx_xp_moe_rows_noalloc(d, 4, 7, p, p, p, p, p, p, p, p, p, p, p, p, p, p, None, p, None, None) == -1
    assert L.tfx_xp_moe_rows_noalloc(d, 4, 0, p, p, p, None, p, p, p, p, p, p, p, p, p, p, None, p, None,
                                     None) == -1  # no ids
    assert L.tfx_xp_moe_rows_noalloc(d, 4, 0, p, p, p, p, p, p, p, p, p, p, p, p, p, p, None, None, None,
                                     None) == -1  # no status
    assert L.tfx_xp_moe_rows_noalloc(d, 200, 0, p, p, p, p, p, p, p, p, p, p, p, p, p, p, None, p, None,
                                     None) == -2  # more than 256 routed pairs
    assert L.tfx_xp_moe_rows_noalloc(d, 0, 0, p, p, p, None, None, p, None, None, p, p, None, None, None, None, None,
                                     p, None, None) == 0  # no rows: nothing to do


def host_entry(lib):
    """The host-buffer layer checks every argument before it queues a copy. Each refused call
    carries a second bad argument, so that one regressed check still queues nothing; R = 0
    queues nothing."""
    L = lib
    d = tfx.dims(7168, 2048, 256, 8)
    p = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    need = L.tfx_xp_moe_rows_host_ws_bytes(d, 1, tfx.ACT_E4M3)
    assert need > 0
    call = lambda dd=d, rows=1, kind=tfx.ACT_E4M3, y=p, status=p, ws=p, wsb=need: L.tfx_xp_moe_rows_host(
        dd, rows, kind, p, p, p, p, p, y, status, None, ws, wsb, None, None)
    assert call(kind=7, status=None) == -1                      # unknown kind
    assert call(ws=ctypes.c_void_p(256 + 16), y=None) == -1     # ws not 256-byte aligned
    assert call(wsb=need - 1, status=None) == -1                # ws too small
    assert call(ws=None, y=None) == -1                          # no ws
    assert call(y=None, status=None) == -1                      # no y_host
    assert call(dd=tfx.dims(7168, 2048, 0, 8), status=None) == -1  # bad sizes
    assert call(rows=33, status=None) == -2                     # 264 routed pairs: beyond the one-launch layer
    assert call(rows=0) == 0                                    # nothing to do


if __name__ == "__main__":
    lib = tfx.load()
    for name in sys.argv[1:]:
        globals()[name](lib)
    print("ok")
