"""The C ABI without a GPU: the library builds, loads and exports every
function include/ep.h declares; the host-only functions (padding, capacity
helpers, workspace sizing, status strings, argument checks) behave as
documented. No kernel is launched here."""
import ctypes as C
import json
import os
import re

import pytest

import combine_topk_ids_expert_gb300 as ep
from combine_topk_ids_expert_gb300 import _abi
from combine_topk_ids_expert_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    build()


def declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if hdr.endswith(".h"):
            src = open(os.path.join(ROOT, "include", hdr)).read()
            names += re.findall(r"^EP_API\s+[\w\s\*]+?\b(ep_\w+)\s*\(", src, re.M)
    return names


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 14
    L = _abi.lib()
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
        assert n in _abi.SIGNATURES, f"{n} has no binding signature"
        assert hasattr(ep, n), f"{n} has no Python binding of the same name"


def test_no_internal_symbols_exported():
    import subprocess
    r = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True,
                       text=True, check=True)
    exported = {line.split()[-1] for line in r.stdout.splitlines() if " T " in line}
    assert exported == set(declared_functions())


def test_pad_tokens_golden():
    g = json.load(open(os.path.join(GOLDEN, "padding_vectors.json")))
    for c in g["single"]:
        assert ep.ep_pad_tokens(c["n"]) == c["padded"]
    for c in g["group"]:
        assert ep.ep_pad_tokens(max(c["counts"])) == c["padded"]
    assert ep.ep_pad_tokens(-1) == -1


def test_capacity_golden():
    g = json.load(open(os.path.join(GOLDEN, "capacity.json")))
    for c in g["pretrain"]:
        assert ep.ep_derive_max_tokens_pretrain(c["local_batch_size"], c["seq_len"], c["cp"],
                                                c["tp"]) == c["expect"]
    for c in g["inference"]:
        assert ep.ep_derive_max_tokens_inference(c["max_num_batched_tokens"], c["cp"],
                                                 c["tp"]) == c["expect"]
    assert ep.ep_validate_max_tokens(4096, 4096) == _abi.EP_OK
    assert ep.ep_validate_max_tokens(0, 1) == _abi.EP_ERR_INVALID_ARG
    assert ep.ep_validate_max_tokens(4095, 4096) == _abi.EP_ERR_CAPACITY


def test_status_strings():
    seen = set()
    for s in range(9):
        msg = ep.ep_status_string(s)
        assert msg and msg != "unknown status"
        seen.add(msg)
    assert len(seen) == 9
    assert ep.ep_status_string(99) == "unknown status"


def cfg(**kw):
    base = dict(num_max_tokens_per_rank=8192, hidden=7168, num_experts=256, num_ranks=8,
                topk=8, dtype=_abi.EP_BF16, num_sms=0, permute_impl=0)
    base.update(kw)
    return _abi.EpConfig(**base)


def test_required_bytes():
    n = ep.ep_buffer_required_bytes(cfg())
    # receive rows R * roundup4(N_max) * K of D bf16, plus scores/src and layout arrays
    rows = 8 * 8192 * 8
    assert n >= rows * 7168 * 2 + rows * 8 + 8192 * 8 * 4
    assert n < rows * 7168 * 2 * 1.01
    assert n % 256 == 0
    assert ep.ep_buffer_required_bytes(cfg(num_max_tokens_per_rank=8190)) == n  # same P
    assert ep.ep_buffer_required_bytes(cfg(num_max_tokens_per_rank=8193)) > n


@pytest.mark.parametrize("bad", [
    dict(num_experts=250),                 # E % R != 0
    dict(topk=0), dict(topk=300),          # K out of range
    dict(num_experts=2048, num_ranks=8),   # E above 1024
    dict(num_ranks=128, num_experts=256),  # R above 64
    dict(hidden=7), dict(hidden=0),        # row bytes not a multiple of 16
    dict(num_max_tokens_per_rank=0),
    dict(dtype=5), dict(permute_impl=9), dict(num_sms=-1), dict(layout_mode=2),
    dict(num_max_tokens_per_rank=1 << 28),  # rows overflow int32
])
def test_required_bytes_rejects(bad):
    assert ep.ep_buffer_required_bytes(cfg(**bad)) == 0


def test_init_rejects_bad_workspace_without_touching_gpu():
    h = C.c_void_p()
    c = cfg()
    L = _abi.lib()
    assert L.ep_buffer_init(C.byref(c), None, 1 << 40, C.byref(h)) == _abi.EP_ERR_WORKSPACE
    assert L.ep_buffer_init(C.byref(c), 0x1000 + 8, 1 << 40, C.byref(h)) == _abi.EP_ERR_WORKSPACE
    assert L.ep_buffer_init(C.byref(c), 0x1000, 16, C.byref(h)) == _abi.EP_ERR_WORKSPACE
    bad = cfg(num_experts=250)
    assert L.ep_buffer_init(C.byref(bad), 0x1000, 1 << 40, C.byref(h)) == _abi.EP_ERR_INVALID_ARG
    assert h.value is None


def test_calls_reject_null_buffer():
    L = _abi.lib()
    assert L.ep_dispatch(None, None, None, None, 0, 0, None, None) == _abi.EP_ERR_INVALID_ARG
    assert L.ep_combine(None, None, None, 0, None, 0, None) == _abi.EP_ERR_INVALID_ARG
    assert L.ep_dispatch_permute(None, None, None, None, None) == _abi.EP_ERR_INVALID_ARG
    assert L.ep_buffer_destroy(None) == _abi.EP_OK


def test_ctypes_mirror_matches_the_header():
    # The ctypes structures and constants of _abi.py against include/ep.h as a C
    # compiler lays them out: every struct's size, every field's offset and size,
    # every EP_* constant's value (a C program generated from the mirror, built by
    # gcc).
    import shutil
    import subprocess
    import tempfile

    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    structs = {"ep_config": _abi.EpConfig, "ep_layout": _abi.EpLayout,
               "ep_dispatch_out": _abi.EpDispatchOut, "ep_dedup_out": _abi.EpDedupOut,
               "ep_buffer_info": _abi.EpBufferInfo}
    consts = sorted(n for n in dir(_abi) if re.fullmatch(r"EP_[A-Z0-9_]+", n))
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ep.h"', "int main(void) {"]
    for cname, st in structs.items():
        lines.append(f'printf("size {cname} %zu\\n", sizeof({cname}));')
        for f, _ in st._fields_:
            lines.append(f'printf("off {cname}.{f} %zu\\n", offsetof({cname}, {f}));')
            lines.append(f'printf("fsz {cname}.{f} %zu\\n", sizeof((({cname}*)0)->{f}));')
    for c in consts:
        lines.append(f'printf("const {c} %lld\\n", (long long)({c}));')
    lines += ["return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "m.c"), os.path.join(d, "m")
        with open(src, "w") as f:
            f.write("\n".join(lines))
        subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                       check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(line.rsplit(" ", 1) for line in out if line)
    for cname, st in structs.items():
        assert int(got[f"size {cname}"]) == C.sizeof(st), cname
        for f, _ in st._fields_:
            assert int(got[f"off {cname}.{f}"]) == getattr(st, f).offset, (cname, f)
            assert int(got[f"fsz {cname}.{f}"]) == getattr(st, f).size, (cname, f)
    for c in consts:
        assert int(got[f"const {c}"]) == getattr(_abi, c), c
