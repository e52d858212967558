"""Build the CPU oracle (test infrastructure only) into oracle/_build/libtfx_oracle.so.

Plain gcc, -ffp-contract=off so every fp32 operation rounds where the source writes it.
Rebuilds when the C source or header is newer than the library.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = [os.path.join(HERE, "tfx_oracle.c")]
HDR = [os.path.join(HERE, "tfx_oracle.h")]
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libtfx_oracle.so")


def control():
    """The planted control the oracle is built with: TFXO_CTL from the environment (tests of
    the pins only), 0 = the oracle as it ships."""
    return int(os.environ.get("TFXO_CTL", "0") or 0)


def build(force=False):
    ctl = control()
    lib = LIB if ctl == 0 else os.path.join(OUT_DIR, "libtfx_oracle_ctl%d.so" % ctl)
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(lib):
        t = os.path.getmtime(lib)
        if all(os.path.getmtime(p) <= t for p in SRC + HDR + [__file__]):
            return lib
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-Wextra", "-DTFXO_CTL=%d" % ctl, "-o", tmp] + SRC + ["-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True))
