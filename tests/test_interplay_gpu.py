"""The dispatch right behind other GPU work on the same stream.

The one-pass dispatch is a cooperative launch whose CTAs meet at a grid
barrier, and it may start early behind the previous kernel (programmatic
dependent launch). A GEMM from the library that fills every SM (a router- or
expert-sized bf16 matmul), then dispatch and combine, repeated: no grid
barrier may run out (the device error word stays clear) and every output
matches the oracle. Also behind the library's own expert GEMM.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_combine_equal, assert_layout_equal, to_dev, to_np

pytestmark = pytest.mark.gpu

T, N, D, E, K, R = 3000, 3000, 4096, 64, 8, 8


def test_dispatch_behind_a_library_matmul(orc):
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16)
    g = torch.Generator(device="cuda").manual_seed(5)
    a = torch.randn((8192, 8192), generator=g, device="cuda", dtype=torch.bfloat16)
    x = W.hidden(190, T, D, "bf16")
    ids, sc = W.routing(190, T, E, K, "zipf", "sigmoid_norm")
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    outs = []
    for _ in range(5):
        c = a @ a                                   # fills every SM for a few ms
        d = buf.dispatch(xd, scd, idd, N)
        outs.append(buf.combine(d.recv_x, scd))
        del c
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    for o in outs:
        assert_combine_equal(to_np(o), want)
    buf.close()


def test_dispatch_behind_the_expert_gemm(orc):
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16)
    x = W.hidden(191, T, D, "bf16")
    ids, sc = W.routing(191, T, E, K, "zipf", "sigmoid_norm")
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    g = torch.Generator(device="cuda").manual_seed(6)
    w = (torch.randn((E, 2048, D), generator=g, device="cuda") * 0.03).to(torch.bfloat16)
    d = buf.dispatch(xd, scd, idd, N)
    outs = []
    for _ in range(4):
        buf.expert_gemm(d.recv_x, w)                # persistent tcgen05 kernel on every SM
        d = buf.dispatch(xd, scd, idd, N)           # may launch while the GEMM drains
        outs.append(buf.combine(d.recv_x, scd))
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    for o in outs:
        assert_combine_equal(to_np(o), want)
    buf.close()
