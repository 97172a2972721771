"""Compile the CPU oracle (plain C, gcc) into a shared library beside this file.

Test infrastructure: the oracle is what the CUDA library is checked against.
``build_oracle(mutant=n)`` builds a deliberately broken copy (n > 0) that the
CPU tests use to show each pin catches a plausible mistake.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ep_oracle.c")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-Wall", "-Wextra"]


# AddressSanitizer build (used by the CPU tests with libasan preloaded).
ASAN_FLAGS = ["-fsanitize=address", "-fno-omit-frame-pointer", "-g"]


def lib_path(mutant: int = 0, sanitize: bool = False) -> str:
    name = "libep_oracle" + ("" if mutant == 0 else f"_mutant{mutant}")
    name += "_asan.so" if sanitize else ".so"
    return os.path.join(HERE, "_build", name)


def build_oracle(mutant: int = 0, force: bool = False, sanitize: bool = False) -> str:
    out = lib_path(mutant, sanitize)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    extra = ASAN_FLAGS if sanitize else []
    cmd = ["gcc", *CFLAGS, *extra, f"-DORACLE_MUTANT={mutant}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
