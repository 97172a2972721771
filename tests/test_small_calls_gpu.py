"""Decode-sized calls of the DeepSeek shape (D = 7168 bf16, E = 256, K = 8, R = 8):
few tokens, so the dispatch counts every id in every CTA instead of meeting at
the grid barrier, and the combine and the dispatch backward spread each token's
row over several CTAs. Every output is compared with the oracle, element by
element, in bf16 and fp32."""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_combine_equal, assert_layout_equal, assert_recv_equal, to_dev, to_np

pytestmark = pytest.mark.gpu

D, E, K, R = 7168, 256, 8, 8


@pytest.mark.parametrize("T", [1, 5, 64, 300, 600])
def test_small_call_matches_oracle(orc, T):
    x = W.hidden(400 + T, T, D, "bf16")
    ids, sc = W.routing(400 + T, T, E, K, "zipf", "sigmoid_norm")
    ids = ids.copy()
    ids[0, -1] = -1                       # a pair routed nowhere
    N = T + 3
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16)
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    out = buf.combine(d.recv_x, scd)
    out32 = buf.combine(d.recv_x, scd, out_dtype=torch.float32)
    S = d.layout.rank_stride
    h = W.normal(500 + T, 1, R * S).astype(np.float32)    # gradient of the receive scores
    gx, gs = buf.dispatch_backward(d.recv_x, T, grad_recv_scores=to_dev(h))
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    for got, kind in ((out, "same"), (out32, "f32")):
        want, err = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R,
                                kind)
        assert err == 0
        assert_combine_equal(to_np(got), want)
    gx_ref, gs_ref, _ = orc.dispatch_backward(ref["recv_x"], h, ref["pos"], ref["rank_prefix"],
                                              ref["S"], R)
    assert np.array_equal(to_np(gx), gx_ref)
    assert np.array_equal(to_np(gs).view(np.uint32), gs_ref.view(np.uint32))
    buf.close()
