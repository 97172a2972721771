"""The C oracle under AddressSanitizer (CPU only).

The real oracle and every deliberately broken copy run all pins in one child
process with libasan preloaded: no out-of-bounds access and no use after free,
whatever a mutant computes. A wrong receive position must be refused with an
error, never written (a write past a buffer would corrupt the test process and
make the CPU suite fail at random). Skipped where gcc has no libasan.
"""
import os
import subprocess
import sys

import pytest

from test_oracle_mutants import MUTANTS

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle
from oracle_pins import PINS
for m in {mutants!r}:
    o = oracle.Oracle(m, sanitize=True)
    for pin in PINS:
        try:
            pin(o)
        except Exception:
            pass
    print("clean", m, flush=True)
"""


def libasan() -> str | None:
    try:
        r = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True,
                           text=True, timeout=30)
    except (OSError, subprocess.TimeoutExpired):
        return None
    path = r.stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_oracle_and_mutants_clean_under_asan():
    lib = libasan()
    if lib is None:
        pytest.skip("gcc has no libasan here")
    mutants = [0] + sorted(MUTANTS)
    env = dict(os.environ, LD_PRELOAD=lib, ASAN_OPTIONS="detect_leaks=0")
    code = CHILD.format(root=ROOT, tests=HERE, mutants=mutants)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    done = [int(line.split()[1]) for line in r.stdout.splitlines() if line.startswith("clean ")]
    assert "AddressSanitizer" not in r.stderr, (
        f"after mutants {done}: {r.stderr[-4000:]}")
    assert r.returncode == 0, r.stderr[-4000:]
    assert done == mutants
