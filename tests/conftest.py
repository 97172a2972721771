import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.get()


@pytest.fixture(params=["onepass", "onepass_barrier", "fused", "vec"])
def path(request, monkeypatch):
    """Each dispatch path in turn: the one-pass cooperative bulk dispatch (the
    default; small calls count every id in every CTA), the same with every call
    meeting at the grid barrier (EP_DISPATCH_SMALL_PAIRS=0), the bulk dispatch as
    count + scan + fused kernels, and the 16-byte vector permute. Returns the
    permute_impl to build the Buffer with."""
    import combine_topk_ids_expert_gb300 as ep
    if request.param == "onepass_barrier":
        monkeypatch.setenv("EP_DISPATCH_SMALL_PAIRS", "0")
    if request.param == "fused":
        monkeypatch.setenv("EP_DISPATCH_ONEPASS", "0")
    return ep.EP_PERMUTE_VEC if request.param == "vec" else ep.EP_PERMUTE_BULK
