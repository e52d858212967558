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
