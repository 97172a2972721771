"""The one-pass dispatch's shared token pool (EP_DISPATCH_POOL, percent of each
tile's tokens that any CTA may copy once its own share is done): whatever the
share, every output equals the oracle's bit for bit. Cases: tiles much longer
than the ring (most of each tile in the pool at 100%), a one-token last tile
that fills its ring from the pool, Zipf routing with pairs routed nowhere, and
the fp32 row type."""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal, to_dev,
                      to_np, torch_dtype)

pytestmark = pytest.mark.gpu

CASES = {
    # name: (seed, T, N, D, dtype, E, K, R, ids)
    "long_tiles": (301, 9001, 9001, 256, "bf16", 64, 4, 4, "zipf"),
    "wide_rows": (302, 6000, 6003, 2048, "bf16", 32, 8, 2, "uniform"),
    "f32": (303, 7000, 7000, 128, "f32", 16, 2, 2, "zipf"),
}


@pytest.mark.parametrize("pool", ["0", "25", "100"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_pool_share_keeps_every_output(orc, monkeypatch, case, pool):
    seed, T, N, D, dtype, E, K, R, ik = CASES[case]
    monkeypatch.setenv("EP_DISPATCH_POOL", pool)
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, ik, "sigmoid_norm")
    ids = ids.copy()
    ids[::97, 0] = -1
    buf = ep.Buffer(N, D, E, R, K, dtype=torch_dtype(dtype))
    scd = to_dev(sc)
    n0 = buf.info()["kernel_launches"]
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    torch.cuda.synchronize()
    assert buf.info()["kernel_launches"] - n0 == 1, "expected the one-pass dispatch"
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    # a second call on the same buffer with other routing: the pool starts over
    ids2, sc2 = W.routing(seed + 1, T, E, K, "uniform", "sigmoid_norm")
    d2 = buf.dispatch(to_dev(x), to_dev(sc2), to_dev(ids2), N)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref2 = orc.dispatch(x, sc2, ids2, N, E, R)
    assert_layout_equal(d2.layout, ref2)
    assert_recv_equal(d2, ref2, R)
    buf.close()
