"""Seeded random shapes: the dispatch paths against the oracle.

24 configurations drawn once from a fixed seed over T, N, N_max, D, dtype, E,
K, R, the id distribution and the layout mode. Each runs the one-pass bulk
dispatch (the default), the three-kernel bulk dispatch (count, scan, fused)
and the vector permute, and compares the layout arrays, every defined receive
row and the combine output with the oracle, bit for bit.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal, to_dev,
                      to_np, torch_dtype)

pytestmark = pytest.mark.gpu


def draw_configs(n: int = 24, seed: int = 0x5EED5, max_recv_bytes: int = 128 << 20):
    """Shapes whose receive buffer (R * roundup4(N_max) * K rows) stays within
    max_recv_bytes, so the oracle's copy fits comfortably on the host."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        R = int(rng.choice([1, 2, 4, 8, 16, 64]))
        E = R * int(rng.choice([1, 2, 3, 8, 16]))
        K = int(rng.integers(1, min(E, 40) + 1))
        T = int(rng.integers(1, 3000))
        N = T + int(rng.integers(0, 6))
        N_max = N + int(rng.integers(0, 9))
        dtype = "bf16" if rng.random() < 0.7 else "f32"
        D = int(rng.choice([8, 16, 24, 64, 200, 512]))
        ids = "zipf" if rng.random() < 0.5 else "uniform"
        layout = "packed" if rng.random() < 0.3 else "strided"
        rows = R * ((N_max + 3) // 4 * 4) * K
        if rows * D * (2 if dtype == "bf16" else 4) > max_recv_bytes:
            continue
        out.append((1000 + len(out), T, N, N_max, D, dtype, E, K, R, ids, layout))
    return out


CONFIGS = draw_configs()
PATHS = ["onepass", "onepass_barrier", "fused", "vec"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cfg", CONFIGS, ids=[f"c{i}" for i in range(len(CONFIGS))])
def test_random_shape(orc, monkeypatch, cfg, path):
    seed, T, N, N_max, D, dtype, E, K, R, ik, layout = cfg
    if path == "fused":
        monkeypatch.setenv("EP_DISPATCH_ONEPASS", "0")
    if path == "onepass_barrier":
        monkeypatch.setenv("EP_DISPATCH_SMALL_PAIRS", "0")
    impl = ep.EP_PERMUTE_VEC if path == "vec" else ep.EP_PERMUTE_BULK
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, ik, "sigmoid_norm")
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=impl, layout=layout)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, N)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    packed = layout == "packed"
    ref = orc.dispatch(x, sc, ids, N, E, R, packed=packed)
    assert_layout_equal(d.layout, ref)
    if packed:
        n = int(ref["rank_prefix"][-1])
        got = to_np(d.recv_x.reshape(-1, D))[:n]
        assert np.array_equal(got, ref["recv_x"][:n])
        assert np.array_equal(to_np(d.recv_src.reshape(-1))[:n], ref["recv_src"][:n])
    else:
        assert_recv_equal(d, ref, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R,
                          packed=packed)
    assert_combine_equal(to_np(out), want)
    buf.close()
