"""The C-ABI library builds for sm_103a, loads, exports every function include/tfx_moe.h
declares, and rejects bad arguments before launching anything (no GPU needed)."""
import os
import re
import shutil
import subprocess
import sys

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


def run_without_device(*cases):
    """Run cases of tests/abi_cases.py in a child process that sees no CUDA device."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="",
               PYTHONPATH=os.pathsep.join([ROOT, os.path.join(ROOT, "tests"), os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "abi_cases.py"), *cases], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.stdout[-3000:], r.stderr[-3000:])


def test_invalid_arguments_are_rejected_before_launch(lib):
    run_without_device("rows_and_route")


def test_chunk_entries_reject_before_launch(lib):
    """The chunk path covers E4M3 activations with H and I multiples of 512 only."""
    run_without_device("chunk")


def test_router_entries_reject_before_launch(lib):
    """Both routers check their sizes, mode and pointers before any launch; R = 0 is a no-op."""
    run_without_device("routers")


def test_noalloc_refuses_before_touching_its_buffer(lib):
    run_without_device("noalloc")


def test_host_entry_refuses_before_queueing(lib):
    run_without_device("host_entry")


def test_host_entry_layout_by_hand(lib):
    """The host entry's input block and workspace, worked out from the widths: the decode layer
    (H 7168, I 2048, 256 experts, top-8, one row, E4M3) and two bf16 rows."""
    from moe_routed_expert_major_gb300 import tfx
    d = tfx.dims(7168, 2048, 256, 8)
    # x 7,168 B; its 224 scales from 7,168; 8 ids from 7,392 (7,392 is 16-aligned); 8 weights
    # from 7,424
    assert tfx.tfx_xp_moe_rows_host_layout(d, 1, tfx.ACT_E4M3) == ([0, 7168, 7392, 7424], 7456)
    # each part at the next 256-byte boundary: counters 4 x (2 + 2 x 256 + 112) = 2,504 B,
    # the inputs 7,456, offs 257 x 4, pair_row and pair_slot 32 each, active 1,024, n_active 4,
    # h 8 x 2,048, its scales 8 x 64, out 8 x 7,168 x 4 and y 7,168 x 2
    sizes = [2504, 7456, 1028, 32, 32, 1024, 4, 16384, 512, 229376, 14336]
    total = 0
    for b in sizes:
        total = (total + b + 255) // 256 * 256
    assert total == 273920
    assert tfx.tfx_xp_moe_rows_host_ws_bytes(d, 1, tfx.ACT_E4M3) == total
    # bf16: x is 2 x 7,168 x 2 B and has no scales, so ids and x_scale share an offset
    assert tfx.tfx_xp_moe_rows_host_layout(d, 2, tfx.ACT_BF16) == ([0, 28672, 28672, 28736], 28800)
    assert tfx.tfx_xp_moe_rows_host_ws_bytes(d, 33, tfx.ACT_E4M3) == 0  # beyond 256 pairs
    assert tfx.tfx_xp_moe_rows_host_ws_bytes(d, 1, 7) == 0

