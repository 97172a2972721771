"""Maximum sizes: the receive buffer at the int32 row limit.

R * S just below 2^31 rows (R = 64 logical ranks, K = E = 64, N_max =
524,284): rank 63's rows start at about 2.11e9 and their byte offsets pass
33 GB, so every position and address computation must hold 64-bit offsets.
The call itself is small (1000 tokens); one token past N_max is rejected.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
from combine_topk_ids_expert_gb300 import _abi
import workloads as W
from gpu_util import assert_combine_equal, assert_layout_equal, to_dev, to_np

pytestmark = pytest.mark.gpu

N_MAX, D, E, R, K, T = 524_284, 4, 64, 64, 64, 1000


def test_positions_and_rows_at_the_int32_edge(orc):
    assert ep.ep_buffer_required_bytes(_abi.EpConfig(N_MAX + 1, D, E, R, K, _abi.EP_F32, 0, 0)) == 0
    x = W.hidden(130, T, D, "f32")
    ids, sc = W.routing(130, T, E, K, "uniform", "sigmoid_norm")   # every token: all 64 experts
    buf = ep.Buffer(N_MAX, D, E, R, K, dtype=torch.float32)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, N_MAX)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.layout(ids, N_MAX, E, R)
    assert_layout_equal(d.layout, ref)
    assert int(ref["pos"].max()) > 2_100_000_000
    pos = d.layout.pos.reshape(-1).long()
    rows = d.recv_x.reshape(-1, D)[pos]
    tok = torch.arange(T, device="cuda").repeat_interleave(K)
    assert torch.equal(rows.view(torch.int32), xd[tok].view(torch.int32))
    # combine of every token against the oracle on a compact copy of its rows
    y = rows.cpu().numpy()                           # [T*K, D]: row t*K+k is pair (t, k)
    cpos = np.arange(T * K, dtype=np.int32).reshape(T, K)
    want, err = orc.combine(y, sc, cpos, np.array([T * K], np.int32), T * K, 1)
    assert err == 0
    assert_combine_equal(to_np(out), want)
    buf.close()
    del buf, d, rows
    torch.cuda.empty_cache()
