"""Per-rank dedupe dispatch and the receiver's expansion, against the oracle.

Every dedupe output (rows, source tokens, local expert indices and scores,
token-rank positions, per-rank totals) is compared bit for bit; the
expansion must reproduce the per-expert dispatch's rows bit for bit, and
combine on the expanded rows must equal combine on the dispatched rows.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_combine_equal, assert_layout_equal, bits, to_dev, to_np, torch_dtype

pytestmark = pytest.mark.gpu

CASES = {
    # name: (seed, T, N, N_max, D, dtype, E, K, R, ids)
    "ds_small":     (120, 1000, 1003, 1024, 256, "bf16", 256, 8, 8, "zipf"),
    "uniform":      (121, 777, 780, 800, 128, "bf16", 64, 4, 4, "uniform"),
    "k1_r1":        (122, 300, 300, 300, 64, "f32", 8, 1, 1, "uniform"),
    "e1024_r64":    (123, 500, 502, 502, 32, "bf16", 1024, 8, 64, "uniform"),
    "tiny_T13":     (124, 13, 16, 32, 64, "f32", 8, 2, 2, "uniform"),
    "k16_r64_odd":  (125, 3001, 3001, 3100, 40, "bf16", 256, 16, 64, "zipf"),
    "prefill_like": (126, 32768, 32768, 32768, 64, "bf16", 256, 8, 8, "zipf"),
}


@pytest.mark.parametrize("form", ["onepass", "fused", "separate"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_dedup_parity_and_expand(orc, monkeypatch, case, form):
    # onepass (the default): one cooperative kernel (layout with a grid
    # barrier, positions, dedupe rows, bulk copies); fused: the same kernel
    # body after separate count and scan kernels; separate: positions, dedupe
    # rows and vector copies as separate kernels
    monkeypatch.setenv("EP_DEDUP_FUSED", "0" if form == "separate" else "1")
    monkeypatch.setenv("EP_DISPATCH_ONEPASS", "1" if form == "onepass" else "0")
    seed, T, N, N_max, D, dtype, E, K, R, ik = CASES[case]
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, ik, "sigmoid_norm")
    ids = ids.copy()
    if T > 3:
        ids[3, 0] = -1
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype))
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    dd = buf.dispatch_dedup(xd, scd, idd, N)
    y = buf.dedup_expand(idd)
    out = buf.combine(y, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch_dedup(x, sc, ids, N, E, R)
    P = ref["P"]
    tir = ref["tokens_in_rank"]
    assert_layout_equal(dd.layout, orc.layout(ids, N, E, R))   # counts, offsets, positions
    assert np.array_equal(to_np(dd.layout.tokens_in_rank), tir)
    assert np.array_equal(to_np(dd.tok_pos), ref["tok_pos"])
    rx = to_np(dd.recv_x.reshape(R * P, D))
    src = to_np(dd.recv_tok_src.reshape(-1))
    idx = to_np(dd.recv_topk_idx.reshape(R * P, K))
    wts = to_np(dd.recv_topk_w.reshape(R * P, K))
    for r in range(R):
        rows = slice(r * P, r * P + int(tir[r]))
        assert np.array_equal(bits(rx[rows]), bits(ref["recv_tok_x"][rows]))
        assert np.array_equal(src[rows], ref["recv_tok_src"][rows])
        assert np.array_equal(idx[rows], ref["recv_topk_idx"][rows])
        assert np.array_equal(wts[rows].view(np.uint32), ref["recv_topk_w"][rows].view(np.uint32))
    # expansion = the per-expert dispatch, and combine agrees
    d = orc.dispatch(x, sc, ids, N, E, R)
    yv = to_np(y.reshape(-1, D))
    valid = d["pos"][d["pos"] >= 0]
    assert np.array_equal(bits(yv[valid]), bits(d["recv_x"][valid]))
    want, _ = orc.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
    assert_combine_equal(to_np(out), want)
    buf.close()


def test_dedup_fullsize_deepseek_matches_dispatch():
    # Full DeepSeek shape: expansion of the dedupe rows equals the per-expert
    # dispatch on every routed row (compared on the device); the dedupe
    # writes ~40% of the rows.
    w = W.WORKLOADS["deepseek"]
    inp = W.make("deepseek")
    xd, idd, scd = to_dev(inp["x"]), to_dev(inp["ids"]), to_dev(inp["scores"])
    a = ep.Buffer(w.N_max, w.D, w.E, w.R, w.K, dtype=torch.bfloat16)
    b = ep.Buffer(w.N_max, w.D, w.E, w.R, w.K, dtype=torch.bfloat16)
    dd = a.dispatch_dedup(xd, scd, idd, w.N)
    y = a.dedup_expand(idd)
    d = b.dispatch(xd, scd, idd, w.N)
    torch.cuda.synchronize()
    assert a.device_error() == 0 and b.device_error() == 0
    pos = d.layout.pos.reshape(-1).long()
    assert torch.equal(y.reshape(-1, w.D)[pos].view(torch.int16),
                       d.recv_x.reshape(-1, w.D)[pos].view(torch.int16))
    rows = int(dd.layout.tokens_in_rank.sum().item())
    assert rows < 0.45 * w.T * w.K
    o1 = a.combine(y, scd)
    o2 = b.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    a.close()
    b.close()
    torch.cuda.empty_cache()


def test_expand_requires_a_dedupe_dispatch():
    buf = ep.Buffer(32, 64, 8, 2, 2, dtype=torch.bfloat16)
    x = to_dev(W.hidden(5, 16, 64, "bf16"))
    ids, sc = W.routing(5, 16, 8, 2, "uniform", "sigmoid_norm")
    buf.dispatch(x, to_dev(sc), to_dev(ids), 16)
    with pytest.raises(ep.EpError) as ei:
        buf.dedup_expand(to_dev(ids))
    assert ei.value.status == ep._abi.EP_ERR_NO_LAYOUT
    buf.dispatch_dedup(x, to_dev(sc), to_dev(ids), 16)
    inside = buf.workspace[:2 * 32 * 2 * 64 * 2].view(torch.bfloat16)   # overlaps recv rows
    with pytest.raises(ep.EpError) as ei:
        ep.ep_dedup_expand(buf.handle, to_dev(ids), inside)
    assert ei.value.status == ep._abi.EP_ERR_INVALID_ARG
    buf.close()
