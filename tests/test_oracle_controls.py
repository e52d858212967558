"""Planted controls: the oracle built with one deliberate mistake (TFXO_CTL = n, see
oracle/tfx_oracle.c) must turn at least one of its pins red, so that the pins are shown to
discriminate. The mistakes are planted in the oracle, on the CPU; TFXO_CTL 0 (the default,
what every other test loads) is the oracle as it ships."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_chain.py", "tests/test_oracle_formats.py", "tests/test_oracle_mass.py"]

CONTROLS = {
    1: "E2M1 nibble order swapped",
    2: "eight-way tree paired differently",
    3: "the first group's scale used for the whole row",
    4: "every group into one accumulator",
    5: "E8M0 weight-scale bias off by one",
    6: "the chain run from the last k down",
    7: "combine slots in reverse order",
    8: "E4M3 ties rounded away from zero",
    9: "mass taken as the magnitude of the sum",
    10: "SwiGLU mass without the g (1 - s) derivative term",
    11: "combine mass with signed weights",
    12: "bf16 of a float64 rounded through binary32",
}


@pytest.mark.parametrize("ctl", sorted(CONTROLS), ids=lambda c: CONTROLS[c].replace(" ", "-"))
def test_pins_catch_planted_mistake(ctl):
    env = dict(os.environ, TFXO_CTL=str(ctl))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", *PINS], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1 and " failed" in r.stdout, (CONTROLS[ctl], r.stdout[-2000:], r.stderr[-2000:])
