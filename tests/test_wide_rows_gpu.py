"""Wide hidden rows on every dispatch path, the combine and the dedupe dispatch.

The bulk dispatch stages whole rows in a shared-memory ring and needs four
slots (two tokens' stores may still be reading the ring while two more rows
load): 32 KB rows leave it six, 40 KB rows five, while 56 KB rows leave too few
and the dispatch falls back to the 16-byte vector kernel, which loops over a
row wider than its CTA's vectors (also 256 KB fp32 rows). Each case is
compared with the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal, bits,
                      to_dev, to_np, torch_dtype)

pytestmark = pytest.mark.gpu

CASES = {
    # name: (seed, T, N, D, dtype, E, K, R)
    "bf16_32k_rows": (170, 61, 64, 16384, "bf16", 8, 2, 2),
    "bf16_40k_rows": (171, 45, 45, 20480, "bf16", 8, 3, 4),
    "bf16_56k_rows": (173, 37, 40, 28672, "bf16", 8, 2, 2),
    "f32_256k_rows": (172, 23, 25, 65536, "f32", 4, 2, 2),
}
# Ring slots the bulk dispatch keeps for each case (0: falls back to the vector kernel).
BULK_STAGES = {"bf16_32k_rows": 6, "bf16_40k_rows": 5, "bf16_56k_rows": 0, "f32_256k_rows": 0}


@pytest.mark.parametrize("case", sorted(CASES))
def test_wide_rows_dispatch_combine(orc, path, case):
    seed, T, N, D, dtype, E, K, R = CASES[case]
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, "zipf", "sigmoid_norm")
    buf = ep.Buffer(N, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=path)
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    info = buf.info()
    if path == ep.EP_PERMUTE_BULK:
        stages = BULK_STAGES[case]
        assert info["permute_impl"] == (ep.EP_PERMUTE_BULK if stages else ep.EP_PERMUTE_VEC)
        assert info["bulk_stages"] == stages
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    buf.close()


@pytest.mark.parametrize("fused", ["1", "0"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_wide_rows_dedup(orc, monkeypatch, case, fused):
    monkeypatch.setenv("EP_DEDUP_FUSED", fused)
    seed, T, N, D, dtype, E, K, R = CASES[case]
    x = W.hidden(seed + 1, T, D, dtype)
    ids, sc = W.routing(seed + 1, T, E, K, "uniform", "sigmoid_norm")
    buf = ep.Buffer(N, D, E, R, K, dtype=torch_dtype(dtype))
    scd, idd = to_dev(sc), to_dev(ids)
    dd = buf.dispatch_dedup(to_dev(x), scd, idd, N)
    y = buf.dedup_expand(idd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch_dedup(x, sc, ids, N, E, R)
    P, tir = ref["P"], ref["tokens_in_rank"]
    rx = to_np(dd.recv_x.reshape(R * P, D))
    for r in range(R):
        rows = slice(r * P, r * P + int(tir[r]))
        assert np.array_equal(bits(rx[rows]), bits(ref["recv_tok_x"][rows]))
    d = orc.dispatch(x, sc, ids, N, E, R)
    valid = d["pos"][d["pos"] >= 0]
    assert np.array_equal(bits(to_np(y.reshape(-1, D))[valid]), bits(d["recv_x"][valid]))
    buf.close()
