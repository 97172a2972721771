"""The one-pass dispatch's grid barrier across many calls on one buffer.

Even and odd barrier generations count their arrivals in separate words, and
each barrier's last arrival zeroes the other word for the next call. Calls of
different sizes launch different numbers of CTAs, so a word left over from an
earlier call, or a generation counted twice, would open a barrier early (a
wrong layout) or never (a timeout). Forty barrier calls in a row, alternating
grid sizes, each compared with the oracle.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_layout_equal, assert_recv_equal, to_dev

pytestmark = pytest.mark.gpu

D, E, K, R = 64, 32, 4, 4
N_MAX = 3000


def test_forty_barrier_calls_of_changing_grid_size(orc, monkeypatch):
    monkeypatch.setenv("EP_DISPATCH_SMALL_PAIRS", "0")   # every call meets at the barrier
    buf = ep.Buffer(N_MAX, D, E, R, K, dtype=torch.bfloat16, permute_impl=ep.EP_PERMUTE_BULK)
    rng = np.random.default_rng(4242)
    # On 152 SMs these sizes launch 3, 17, 150, 151, 152, 77, 140 and 150 CTAs
    # (one tile per CTA, ceil(T / 152) tokens per tile).
    for i in range(40):
        T = int(rng.choice([3, 17, 150, 151, 152, 153, 700, 2999, 3000]))
        x = W.hidden(6000 + i, T, D, "bf16")
        ids, sc = W.routing(6000 + i, T, E, K, "zipf" if i % 2 else "uniform", "sigmoid_norm")
        n0 = buf.info()["kernel_launches"]
        d = buf.dispatch(to_dev(x), to_dev(sc), to_dev(ids), T)
        torch.cuda.synchronize()
        assert buf.info()["kernel_launches"] - n0 == 1, "expected the one-pass dispatch"
        assert buf.device_error() == 0, (i, T)
        ref = orc.dispatch(x, sc, ids, T, E, R)
        assert_layout_equal(d.layout, ref)
        assert_recv_equal(d, ref, R)
    buf.close()
