"""The token-slice form of the oracle that the full-size GPU tests use equals
the oracle run on the whole call: combine (bf16 and fp32) and backward, on
small calls with several slices, a ragged last slice, pairs routed nowhere and
a token with no expert at all."""
import numpy as np
import pytest

import workloads as W
from gpu_util import oracle_backward_all, oracle_combine_all


def _case(seed, T, N, D, E, K, R):
    x = W.hidden(seed, T, D, "bf16")
    ids, sc = W.routing(seed, T, E, K, "zipf", "sigmoid_norm")
    ids = ids.copy()
    ids[1, 0] = -1
    ids[T - 1, :] = -1
    return x, ids, sc, N, E, R


@pytest.mark.parametrize("chunk", [7, 64, 1000])
def test_slices_equal_the_whole_call(orc, chunk):
    x, ids, sc, N, E, R = _case(3, 150, 153, 32, 16, 4, 4)
    d = orc.dispatch(x, sc, ids, N, E, R)
    for kind in ("same", "f32"):
        want, _ = orc.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R, kind)
        got = oracle_combine_all(orc, x, sc, d["pos"], kind, chunk=chunk)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), kind
    g = W.hidden(4, x.shape[0], x.shape[1], "bf16")
    gy, gs, _ = orc.combine_backward(g, d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
    gx, _, _ = orc.dispatch_backward(gy, None, d["pos"], d["rank_prefix"], d["S"], R)
    gy_s, gs_s, gx_s = oracle_backward_all(orc, x, g, sc, d["pos"], chunk=chunk)
    p = d["pos"].ravel()
    assert np.array_equal(gy_s, gy[p[p >= 0]])
    assert np.array_equal(gs_s.view(np.uint32), gs.view(np.uint32))
    assert np.array_equal(gx_s, gx)
