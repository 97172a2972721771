"""Degenerate cases of the method against the oracle, on every dispatch path.

- one expert, one rank, top-1, one token, the smallest row (16 bytes);
- no routing at all (every id is -1): empty layout, zero output rows;
- K = E: every token selects every expert;
- a tiny call in a large buffer (T = 1 with N_max = 100,000: the per-rank
  stride follows the call's N, not N_max);
- the combine follows ascending k (an order-sensitive fma chain);
- an empty call (T = 0) after a full one: the layout describes the empty call.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal, to_dev,
                      to_np, torch_dtype)

pytestmark = pytest.mark.gpu


def check(orc, x, ids, sc, N, N_max, D, dtype, E, K, R, impl):
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=impl)
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert buf.device_error() == ref["err"]
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    buf.close()
    return ref, to_np(out)


def test_one_expert_one_token_smallest_row(orc, path):
    x = W.hidden(150, 1, 8, "bf16")
    ids = np.zeros((1, 1), np.int32)
    sc = np.full((1, 1), 0.75, np.float32)
    ref, out = check(orc, x, ids, sc, 1, 1, 8, "bf16", 1, 1, 1, path)
    assert int(ref["rank_prefix"][-1]) == 1 and ref["S"] == 4   # P = roundup4(1) = 4


def test_no_routing_at_all(orc, path):
    T, D, E, K, R = 300, 64, 16, 4, 4
    x = W.hidden(151, T, D, "f32")
    ids = np.full((T, K), -1, np.int32)
    sc = W.routing(151, T, E, K, "uniform", "sigmoid_norm")[1]
    ref, out = check(orc, x, ids, sc, T, T, D, "f32", E, K, R, path)
    assert int(ref["rank_prefix"][-1]) == 0
    assert np.all(out == 0)


def test_every_token_selects_every_expert(orc, path):
    T, D, E, R = 257, 128, 8, 2
    x = W.hidden(152, T, D, "bf16")
    ids, sc = W.routing(152, T, E, E, "uniform", "softmax_topk")
    ref, _ = check(orc, x, ids, sc, T, T, D, "bf16", E, E, R, path)
    assert np.all(ref["cnt"] == T)


def test_tiny_call_in_a_large_buffer(orc, path):
    x = W.hidden(153, 1, 64, "bf16")
    ids, sc = W.routing(153, 1, 32, 4, "uniform", "sigmoid_norm")
    ref, _ = check(orc, x, ids, sc, 1, 100_000, 64, "bf16", 32, 4, 8, path)
    assert ref["S"] == 4 * 4


def test_combine_follows_ascending_k(orc, path):
    # Scores (1, 2^-24, -1) on rows of ones: the fp32 fma chain in ascending k
    # gives exactly +0 (1, then a tie rounded to even, then 0); any other order
    # gives 2^-24. Checked for two orders of the same experts.
    for order in ([0, 1, 2], [2, 0, 1]):
        x = np.ones((1, 4), np.float32)
        ids = np.array([order], np.int32)
        sc = np.array([[1.0, 2.0 ** -24, -1.0]], np.float32)
        _, out = check(orc, x, ids, sc, 1, 1, 4, "f32", 4, 3, 1, path)
        assert np.array_equal(out.view(np.uint32), np.zeros((1, 4), np.uint32))


def test_empty_call_after_a_full_one(orc, path):
    # T = 0 (with N = 0 and with N = 6) after a call that filled the layout: the
    # layout must describe the empty call (every count and prefix zero, S = P*K),
    # not the previous one; the combine of zero tokens is a no-op; the next full
    # call is exact again.
    D, E, K, R = 64, 16, 4, 4
    buf = ep.Buffer(300, D, E, R, K, dtype=torch.bfloat16, permute_impl=path)
    x = W.hidden(154, 200, D, "bf16")
    ids, sc = W.routing(154, 200, E, K, "zipf", "sigmoid_norm")
    buf.dispatch(to_dev(x), to_dev(sc), to_dev(ids), 200)
    for N in (0, 6):
        x0 = np.zeros((0, D), np.uint16)
        ids0 = np.zeros((0, K), np.int32)
        sc0 = np.zeros((0, K), np.float32)
        d = buf.dispatch(to_dev(x0), to_dev(sc0), to_dev(ids0), N)
        out = buf.combine(d.recv_x, to_dev(sc0))
        torch.cuda.synchronize()
        assert buf.device_error() == 0
        assert out.shape == (0, D)
        ref = orc.dispatch(x0, sc0, ids0, N, E, R)
        assert_layout_equal(d.layout, ref)
        assert ref["S"] == ((N + 3) // 4 * 4) * K
    check(orc, x, ids, sc, 200, 300, D, "bf16", E, K, R, path)
