"""The per-rank token counts printed on "fix(moe): equalize and align per-rank
token counts for HybridEP dispatch" ("Problem", "Testing" and the nightly A/B
table), run through the GPU dispatch and combine.

For every count n of the fixture, a call with T = N = n must use the padded
count the page's rule gives (the fixture's hand-worked value) as its capacity:
S = padded * K. For every group of counts (the functional test's combos and
the DeepSeek-V4-Flash row), each member runs with T = its own count and N = the
group max; the layout, receive rows and combine match the oracle bit for bit,
and ("Testing": unequal runs reproduce the equal-count run) the combined output
equals the same tokens dispatched with N = T.
"""
import json
import os

import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal, bits,
                      to_dev, to_np)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "padding_vectors.json")
D, E, K, R = 64, 32, 4, 4


def fixture():
    with open(GOLDEN) as f:
        return json.load(f)


def run(orc, buf, seed, T, N):
    x = W.hidden(seed, T, D, "bf16")
    ids, sc = W.routing(seed, T, E, K, "zipf", "sigmoid_norm")
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    got = to_np(out)
    assert_combine_equal(got, want)
    return d.layout.rank_stride, got


def test_single_counts_pad_to_the_worked_values(orc):
    buf = ep.Buffer(4096, D, E, R, K, dtype=torch.bfloat16)
    for i, c in enumerate(fixture()["single"]):
        S, _ = run(orc, buf, 180 + i, c["n"], c["n"])
        assert S == c["padded"] * K, (c["n"], S, c["cite"])
    buf.close()


def test_groups_pad_to_the_group_max_and_match_equal_runs(orc):
    buf = ep.Buffer(4096, D, E, R, K, dtype=torch.bfloat16)
    for g_i, g in enumerate(fixture()["group"]):
        N = max(g["counts"])
        for r_i, T in enumerate(g["counts"]):
            seed = 300 + 20 * g_i + r_i
            S, out_group = run(orc, buf, seed, T, N)
            assert S == g["padded"] * K, (g["counts"], S, g["cite"])
            _, out_alone = run(orc, buf, seed, T, T)
            assert np.array_equal(bits(out_group), bits(out_alone)), (g["counts"], T)
    buf.close()
