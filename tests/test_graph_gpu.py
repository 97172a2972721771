"""CUDA-graph capture and replay of layout -> dispatch -> expert -> combine.

The sequence is captured once and replayed with fresh routing written into
the captured input buffers; each replay is checked against the oracle and
against eager calls, and eager calls of another size are interleaved on the
same buffer between replays (the pages' test_ht_cudagraph.py design: fresh
routing per replay, analytic oracle plus eager comparison, eager/replay
interleave on one Buffer).
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal,
                      oracle_combine_all, to_dev, to_np)

pytestmark = pytest.mark.gpu


def expert_standin(recv_x, recv_src, ids_flat, y):
    """y = 2^((e mod 4) - 1) * recv_x with e the row's expert (exact in bf16).
    Rows past a rank's total carry garbage sources: clamped, never combined."""
    src = recv_src.reshape(-1).clamp(0, ids_flat.numel() - 1).long()
    e = ids_flat[src].long()
    scale = torch.exp2(((e % 4) - 1).float())
    y.copy_((recv_x.reshape(y.shape).float() * scale[:, None]).to(y.dtype))


def oracle_scaled(orc, x, sc, ids, N, E, R):
    ref = orc.dispatch(x, sc, ids, N, E, R)
    y = ref["recv_x"].copy()
    T, K = ids.shape
    for t in range(T):
        for k in range(K):
            p = ref["pos"][t, k]
            v = (y[p].astype(np.uint32) << 16).view(np.float32) * np.float32(
                2.0 ** ((ids[t, k] % 4) - 1))
            y[p] = (v.view(np.uint32) >> 16).astype(np.uint16)
    out, _ = orc.combine(y, sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    return ref, out


@pytest.mark.parametrize("impl", [ep.EP_PERMUTE_VEC, ep.EP_PERMUTE_BULK], ids=["vec", "bulk"])
def test_graph_replay_fresh_routing_and_interleave(orc, impl):
    T, N, D, E, K, R = 1000, 1003, 256, 256, 8, 8
    N_max = 1024
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch.bfloat16, permute_impl=impl)
    S = ep.ep_pad_tokens(N) * K
    x = W.hidden(31, T, D, "bf16")
    xd = to_dev(x)
    ids_d = torch.empty((T, K), dtype=torch.int32, device="cuda")
    sc_d = torch.empty((T, K), dtype=torch.float32, device="cuda")
    y = torch.empty((R * S, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")

    def seq(stream):
        d = buf.dispatch(xd, sc_d, ids_d, N, stream=stream)
        expert_standin(d.recv_x, d.recv_src, ids_d.reshape(-1), y)
        buf.combine(y, sc_d, out=out, stream=stream)
        return d

    ids0, sc0 = W.routing(40, T, E, K, "zipf", "sigmoid_norm")
    ids_d.copy_(torch.from_numpy(ids0))
    sc_d.copy_(torch.from_numpy(sc0))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        seq(s)                                     # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        d_cap = seq(s)
    torch.cuda.synchronize()

    for i in range(12):
        ids_i, sc_i = W.routing(41 + i, T, E, K, "zipf", "sigmoid_norm")
        ids_d.copy_(torch.from_numpy(ids_i))
        sc_d.copy_(torch.from_numpy(sc_i))
        g.replay()
        torch.cuda.synchronize()
        ref, want = oracle_scaled(orc, x, sc_i, ids_i, N, E, R)
        assert_layout_equal(d_cap.layout, ref)
        assert_recv_equal(d_cap, ref, R)
        assert_combine_equal(to_np(out), want)
        assert buf.device_error() == 0
        replay_out = out.clone()
        # eager call of the same inputs on the same buffer: identical bits
        seq(torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), replay_out.view(torch.int16))
        # eager call of another size in between replays (prefill-eager / decode-graphed)
        T2 = 37 + 3 * i
        ids2, sc2 = W.routing(90 + i, T2, E, K, "uniform", "sigmoid_norm")
        x2 = W.hidden(90 + i, T2, D, "bf16")
        d2 = buf.dispatch(to_dev(x2), to_dev(sc2), to_dev(ids2), T2 + 2)
        o2 = buf.combine(d2.recv_x, to_dev(sc2))
        torch.cuda.synchronize()
        ref2 = orc.dispatch(x2, sc2, ids2, T2 + 2, E, R)
        assert_layout_equal(d2.layout, ref2)
        want2, _ = orc.combine(ref2["recv_x"], sc2, ref2["pos"], ref2["rank_prefix"], ref2["S"], R)
        assert_combine_equal(to_np(o2), want2)
    buf.close()


def test_prefill32k_graph_100_replays(orc):
    # 32k-token prefill in worst-token graph mode: one capture, 100 replays
    # with fresh Zipf(1.1) routing. Counts and positions are checked against
    # the oracle on every replay; on replays 0, 1, 49, 98, 99 every receive row
    # and the combine of every token, in bf16 and in fp32 before the cast, are
    # checked against the oracle, and the replay equals an eager run.
    w = W.WORKLOADS["prefill32k"]
    T, N, D, E, K, R = w.T, w.N, w.D, w.E, w.K, w.R
    buf = ep.Buffer(w.N_max, D, E, R, K, dtype=torch.bfloat16)
    x = W.hidden(w.seed, T, D, "bf16")
    xd = to_dev(x)
    ids_d = torch.empty((T, K), dtype=torch.int32, device="cuda")
    sc_d = torch.empty((T, K), dtype=torch.float32, device="cuda")
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty((T, D), dtype=torch.float32, device="cuda")
    inp0 = W.make("prefill32k", replay=0, with_x=False)
    ids_d.copy_(torch.from_numpy(inp0["ids"]))
    sc_d.copy_(torch.from_numpy(inp0["scores"]))

    def seq(stream):
        d = buf.dispatch(xd, sc_d, ids_d, N, stream=stream)
        buf.combine(d.recv_x, sc_d, out=out, stream=stream)
        buf.combine(d.recv_x, sc_d, out=out32, out_dtype=torch.float32, stream=stream)
        return d

    g, d = _capture(seq)
    eager = ep.Buffer(w.N_max, D, E, R, K, dtype=torch.bfloat16)
    full = {0, 1, 49, 98, 99}
    for i in range(w.graph_replays):
        inp = W.make("prefill32k", replay=i, with_x=False)
        ids_d.copy_(torch.from_numpy(inp["ids"]))
        sc_d.copy_(torch.from_numpy(inp["scores"]))
        g.replay()
        torch.cuda.synchronize()
        ref = orc.layout(inp["ids"], N, E, R)
        assert_layout_equal(d.layout, ref)
        if i in full:
            pos = d.layout.pos.reshape(-1).long()
            rows = d.recv_x.reshape(-1, D)[pos].view(torch.int16)
            tok = torch.arange(T, device="cuda").repeat_interleave(K)
            assert torch.equal(rows, xd[tok].view(torch.int16))
            del rows, tok
            for got, kind in ((out, "same"), (out32, "f32")):
                want = oracle_combine_all(orc, x, inp["scores"], ref["pos"], kind)
                assert_combine_equal(to_np(got), want)
                del want
            de = eager.dispatch(xd, sc_d, ids_d, N)
            oe = eager.combine(de.recv_x, sc_d)
            torch.cuda.synchronize()
            assert torch.equal(oe.view(torch.int16), out.view(torch.int16))
            del de, oe
    assert buf.device_error() == 0
    buf.close()
    eager.close()
    torch.cuda.empty_cache()


def _capture(seq):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        seq(s)                                     # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        res = seq(s)
    torch.cuda.synchronize()
    return g, res


def test_graph_dedupe_path_fresh_routing(orc):
    # The per-rank dedupe dispatch, the receiver's expansion and the combine,
    # captured once and replayed with fresh routing: every replay matches the
    # oracle (dedupe rows, expansion, combine).
    T, N, D, E, K, R = 700, 702, 128, 64, 8, 8
    buf = ep.Buffer(704, D, E, R, K, dtype=torch.bfloat16)
    x = W.hidden(60, T, D, "bf16")
    xd = to_dev(x)
    ids_d = torch.empty((T, K), dtype=torch.int32, device="cuda")
    sc_d = torch.empty((T, K), dtype=torch.float32, device="cuda")
    S = ep.ep_pad_tokens(N) * K
    y = torch.empty((R, S, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")

    def seq(stream):
        dd = buf.dispatch_dedup(xd, sc_d, ids_d, N, stream=stream)
        buf.dedup_expand(ids_d, y_recv=y, stream=stream)
        buf.combine(y, sc_d, out=out, stream=stream)
        return dd

    ids0, sc0 = W.routing(61, T, E, K, "zipf", "sigmoid_norm")
    ids_d.copy_(torch.from_numpy(ids0))
    sc_d.copy_(torch.from_numpy(sc0))
    g, dd = _capture(seq)
    for i in range(6):
        ids_i, sc_i = W.routing(62 + i, T, E, K, "zipf" if i % 2 else "uniform", "sigmoid_norm")
        ids_d.copy_(torch.from_numpy(ids_i))
        sc_d.copy_(torch.from_numpy(sc_i))
        g.replay()
        torch.cuda.synchronize()
        assert buf.device_error() == 0
        ref = orc.dispatch_dedup(x, sc_i, ids_i, N, E, R)
        P, tir = ref["P"], ref["tokens_in_rank"]
        rx = to_np(dd.recv_x.reshape(R * P, D))
        for r in range(R):
            rows = slice(r * P, r * P + int(tir[r]))
            assert np.array_equal(rx[rows], ref["recv_tok_x"][rows]), (i, r)
        d = orc.dispatch(x, sc_i, ids_i, N, E, R)
        valid = d["pos"][d["pos"] >= 0]
        assert np.array_equal(to_np(y.reshape(-1, D))[valid], d["recv_x"][valid])
        want, _ = orc.combine(d["recv_x"], sc_i, d["pos"], d["rank_prefix"], d["S"], R)
        assert_combine_equal(to_np(out), want)
    buf.close()


def test_graph_backward_fresh_routing(orc):
    # Dispatch, combine backward and dispatch backward captured once and
    # replayed with fresh routing and a fresh upstream gradient.
    T, N, D, E, K, R = 600, 600, 256, 32, 4, 4
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16)
    x = W.hidden(70, T, D, "bf16")
    xd = to_dev(x)
    ids_d = torch.empty((T, K), dtype=torch.int32, device="cuda")
    sc_d = torch.empty((T, K), dtype=torch.float32, device="cuda")
    g_d = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    S = ep.ep_pad_tokens(N) * K
    grad_y = torch.empty((R, S, D), dtype=torch.bfloat16, device="cuda")
    state = {}

    def seq(stream):
        d = buf.dispatch(xd, sc_d, ids_d, N, stream=stream)
        buf.combine_backward(g_d, d.recv_x, sc_d, grad_y=grad_y, want_scores=False,
                             stream=stream)
        gx, _ = buf.dispatch_backward(grad_y, T, stream=stream)
        state["gx"] = gx
        return d

    ids0, sc0 = W.routing(71, T, E, K, "uniform", "sigmoid_norm")
    ids_d.copy_(torch.from_numpy(ids0))
    sc_d.copy_(torch.from_numpy(sc0))
    g_d.copy_(to_dev(W.hidden(72, T, D, "bf16")))
    g, _ = _capture(seq)
    gx = state["gx"]
    for i in range(5):
        ids_i, sc_i = W.routing(73 + i, T, E, K, "zipf", "sigmoid_norm")
        gi = W.hidden(80 + i, T, D, "bf16")
        ids_d.copy_(torch.from_numpy(ids_i))
        sc_d.copy_(torch.from_numpy(sc_i))
        g_d.copy_(to_dev(gi))
        g.replay()
        torch.cuda.synchronize()
        assert buf.device_error() == 0
        ref = orc.dispatch(x, sc_i, ids_i, N, E, R)
        gy_ref, _, _ = orc.combine_backward(gi, ref["recv_x"], sc_i, ref["pos"],
                                            ref["rank_prefix"], ref["S"], R)
        valid = ref["pos"][ref["pos"] >= 0]
        assert np.array_equal(to_np(grad_y.reshape(-1, D))[valid], gy_ref[valid]), i
        gx_ref, _, _ = orc.dispatch_backward(gy_ref, None, ref["pos"], ref["rank_prefix"],
                                             ref["S"], R)
        assert np.array_equal(to_np(gx), gx_ref), i
    buf.close()
