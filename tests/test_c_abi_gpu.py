"""The C ABI used from plain C: tests/c/abi_roundtrip.c is compiled with gcc
against include/ep.h, linked with libep_gb300 and, separately, the oracle's
library, and run: one dispatch + combine must match the oracle bit for bit."""
import os
import subprocess

import pytest

from combine_topk_ids_expert_gb300.build import build as build_lib
from oracle.build import build_oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_program_matches_the_oracle(tmp_path):
    lib = build_lib()
    orc = build_oracle()
    exe = str(tmp_path / "abi_roundtrip")
    lib_dir, orc_dir = os.path.dirname(lib), os.path.dirname(orc)
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", os.path.join(ROOT, "tests", "c", "abi_roundtrip.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-lep_gb300", "-L", orc_dir, "-lep_oracle",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}:{orc_dir}:{os.path.join(CUDA, 'lib64')}", "-o", exe]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c-abi ok" in r.stdout
