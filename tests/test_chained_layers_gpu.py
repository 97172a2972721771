"""Layers chained on one stream with no synchronisation: each layer's combine
output is the next layer's dispatch input (x), as in a stack of MoE layers.

The dispatch may start while the combine before it drains (programmatic
dependent launch); it must still read the combine's finished rows. Every
layer's receive buffers and output are compared with the oracle run on the
oracle's own previous output, so a row read before the combine wrote it shows
up as a mismatch in that layer or the next.
"""
from types import SimpleNamespace

import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_combine_equal, assert_recv_equal, to_dev, to_np, torch_dtype

pytestmark = pytest.mark.gpu

LAYERS = 4

CASES = {
    # name: (T, N, D, E, K, R, dtype) -- the grid-barrier path (many tiles, token
    # pool) and the small-call path (at most 2048 pairs) of the one-pass dispatch
    "barrier_bf16": (2000, 2003, 1024, 64, 8, 8, "bf16"),
    "barrier_f32": (1500, 1500, 512, 32, 4, 4, "f32"),
    "small_bf16": (200, 203, 7168, 256, 8, 8, "bf16"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_combine_output_feeds_next_dispatch(orc, path, case):
    T, N, D, E, K, R, dtype = CASES[case]
    buf = ep.Buffer(N, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=path)
    x0 = W.hidden(9100 + T, T, D, dtype)
    routes = [W.routing(9200 + 10 * l + T, T, E, K, "zipf" if l % 2 else "uniform",
                        "sigmoid_norm") for l in range(LAYERS)]
    dev_routes = [(to_dev(ids), to_dev(sc)) for ids, sc in routes]
    torch.cuda.synchronize()
    # Every layer on the current stream, no host synchronisation in between.
    xd = to_dev(x0)
    got = []
    for idd, scd in dev_routes:
        d = buf.dispatch(xd, scd, idd, N)
        recv = tuple(t.clone() for t in (d.recv_x, d.recv_scores, d.recv_src))
        xd = buf.combine(d.recv_x, scd)
        got.append((recv, d.layout, xd))
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    # The oracle chain: layer l's input is the oracle's own output of layer l-1.
    x = x0
    for (ids, sc), ((rx, rs, rsrc), lay, out) in zip(routes, got):
        ref = orc.dispatch(x, sc, ids, N, E, R)
        assert_recv_equal(SimpleNamespace(recv_x=rx, recv_scores=rs, recv_src=rsrc,
                                          layout=lay), ref, R)
        x, err = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
        assert err == 0
        assert_combine_equal(to_np(out), x)
    buf.close()
