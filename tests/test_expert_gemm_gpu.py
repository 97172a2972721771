"""The tcgen05 grouped GEMM (expert consumer) against the oracle.

y[p] = x[p] * W_e^T over each expert's receive rows, driven by the device
counts of the last dispatch. The tensor cores' summation order is the
hardware's, so each output is compared with the oracle's value (fp64 sum,
one bf16 rounding) within |gpu - oracle| <= 2^-7 max(|gpu|, |oracle|) +
2 din 2^-24 m, m = sum_i |x_i w_i|: the fp32 summation bound, plus one bf16
ulp because the two sides round different sums and may land on neighbours.
Rows that belong to no expert must keep their contents.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import pool_map, assert_combine_equal, to_dev, to_np

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC1   # a bf16 NaN pattern no GEMM output produces


def f32(h):
    return (h.astype(np.uint32) << 16).view(np.float32)


def check_gemm(orc, y_gpu, x_ref, w, cnt, off):
    y_ref = orc.expert_gemm(x_ref, w, cnt, off, fill=SENTINEL)
    xf, wf = np.abs(f32(x_ref).astype(np.float64)), np.abs(f32(w).astype(np.float64))
    din = w.shape[2]
    covered = np.zeros(y_ref.shape[0], bool)
    for e in range(w.shape[0]):
        lo, n = int(off[e]), int(cnt[e])
        if n == 0:
            continue
        covered[lo:lo + n] = True
        g = f32(y_gpu[lo:lo + n]).astype(np.float64)
        r = f32(y_ref[lo:lo + n]).astype(np.float64)
        mag = xf[lo:lo + n] @ wf[e].T
        tol = 2.0 ** -7 * np.maximum(np.abs(r), np.abs(g)) + 2.0 * din * 2.0 ** -24 * mag + 1e-30
        bad = np.abs(g - r) > tol
        assert not bad.any(), (f"expert {e}: {int(bad.sum())} outputs outside the bound, "
                               f"e.g. gpu {g[bad][:4]} oracle {r[bad][:4]} tol {tol[bad][:4]}")
    assert np.all(y_gpu[~covered] == SENTINEL), "rows of no expert were written"


CASES = {
    # name: (seed, T, N, din, dout, E, K, R, ids, layout)
    "bn256_zipf":   (70, 300, 300, 256, 256, 16, 4, 4, "zipf", "strided"),
    "bn128":        (71, 250, 252, 128, 128, 8, 2, 2, "uniform", "strided"),
    "bn128_384":    (72, 180, 180, 192, 384, 8, 2, 1, "uniform", "strided"),
    "packed":       (73, 300, 301, 256, 256, 16, 4, 4, "zipf", "packed"),
    "ds_like":      (74, 1000, 1003, 1024, 512, 32, 8, 8, "zipf", "strided"),
    "many_empty":   (75, 37, 40, 128, 256, 256, 8, 8, "uniform", "strided"),
    # more cases on the 2-SM kernel (dout % 256 == 0): 256-row tiles, odd and
    # even tile counts per expert, empty experts, the packed layout
    "pair_zipf":    (76, 600, 600, 256, 512, 16, 4, 4, "zipf", "strided"),
    "pair_packed":  (77, 500, 503, 128, 1024, 8, 2, 2, "uniform", "packed"),
    "pair_empty":   (78, 37, 40, 64, 512, 256, 8, 8, "uniform", "strided"),
    "pair_e1024":   (79, 300, 300, 64, 512, 1024, 8, 64, "uniform", "strided"),
    "pair_big":     (82, 2000, 2000, 512, 2048, 8, 2, 2, "zipf", "strided"),
}


def expected_kind(kind: str, dout: int) -> int:
    return int(kind) if dout % 256 == 0 else 1


@pytest.mark.parametrize("kind,bk,light", [("2", "64", None), ("1", "64", None), ("2", "32", None),
                                           ("1", "64", "0"), ("2", "64", "0")])
@pytest.mark.parametrize("case", sorted(CASES))
def test_expert_gemm_parity(orc, monkeypatch, case, kind, bk, light):
    # kind: 1 single-CTA 128-row tiles, 2 two-SM 256-row tiles (falls back to 1
    # where dout % 256 != 0); bk: K per ring stage (128-byte swizzle at 64,
    # 64-byte at 32); light: the schedule's light-expert threshold in rows
    # (None: the default, light experts interleaved with heavy ones; "0": one
    # sequence in expert order)
    monkeypatch.setenv("EP_GEMM_KERNEL", kind)
    monkeypatch.setenv("EP_GEMM_BK", bk)
    if light is None:
        monkeypatch.delenv("EP_GEMM_LIGHT_ROWS", raising=False)
    else:
        monkeypatch.setenv("EP_GEMM_LIGHT_ROWS", light)
    seed, T, N, din, dout, E, K, R, ik, layout = CASES[case]
    x = W.hidden(seed, T, din, "bf16")
    ids, sc = W.routing(seed, T, E, K, ik, "sigmoid_norm")
    w = W.hidden(seed + 1, E * dout, din, "bf16").reshape(E, dout, din)
    buf = ep.Buffer(N, din, E, R, K, dtype=torch.bfloat16, layout=layout)
    d = buf.dispatch(to_dev(x), to_dev(sc), to_dev(ids), N)
    S = d.layout.rank_stride
    y = torch.full((R * S, dout), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    buf.expert_gemm(d.recv_x.reshape(R * S, din), to_dev(w), y_recv=y)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    assert buf.info()["gemm_kernel"] == expected_kind(kind, dout)
    ref = orc.dispatch(x, sc, ids, N, E, R, packed=(layout == "packed"))
    check_gemm(orc, to_np(y), ref["recv_x"], w, ref["cnt"], ref["expert_offset"])
    buf.close()


@pytest.mark.parametrize("name", ["deepseek", "mixtral"])
def test_gemm_variants_fullsize(orc, monkeypatch, name):
    # Full workload shape, D -> 2048: the 2-SM kernel (M = 256 across a pair)
    # and the single-CTA kernel (M = 128), at 64- and 32-wide K slices, issue the
    # same K=16 steps in the same order for every output, so all agree bit for
    # bit; so do the schedules (light experts interleaved with heavy ones at the
    # default threshold, none light, all light), which change only which SM
    # computes a tile and when. Every row of the hottest, the median and the
    # coldest expert is checked against the oracle.
    w_ = W.WORKLOADS[name]
    inp = W.make(name)
    D, E, dout = w_.D, w_.E, 2048
    xd, idd, scd = to_dev(inp["x"]), to_dev(inp["ids"]), to_dev(inp["scores"])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    wd = (torch.randn((E * dout, D), generator=gen, device="cuda") * 0.03).to(torch.bfloat16)
    bufs, ys = [], []
    for kind, bk, light in (("2", "64", None), ("1", "64", None), ("2", "32", None),
                            ("1", "32", None), ("1", "64", "0"), ("2", "64", "0"),
                            ("1", "64", "1000000"), ("2", "64", "1000000")):
        monkeypatch.setenv("EP_GEMM_KERNEL", kind)
        monkeypatch.setenv("EP_GEMM_BK", bk)
        if light is None:
            monkeypatch.delenv("EP_GEMM_LIGHT_ROWS", raising=False)
        else:
            monkeypatch.setenv("EP_GEMM_LIGHT_ROWS", light)
        buf = ep.Buffer(w_.N_max, D, E, w_.R, w_.K, dtype=torch.bfloat16)
        d = buf.dispatch(xd, scd, idd, w_.N)
        rows = w_.R * d.layout.rank_stride
        y = torch.full((rows, dout), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        buf.expert_gemm(d.recv_x.reshape(rows, D), wd.reshape(E, dout, D), y_recv=y)
        torch.cuda.synchronize()
        assert buf.device_error() == 0
        assert buf.info()["gemm_kernel"] == int(kind)
        if bufs:
            buf.close()
            assert torch.equal(ys[0].view(torch.int16), y.view(torch.int16)), (kind, bk, light)
            del d, y
        else:
            bufs.append((buf, d))
            ys.append(y)
    buf, d = bufs[0]
    # Every row of the hottest, the median and the coldest used expert against
    # the oracle, with each row's input taken from x through the oracle's own
    # layout (receive row pos[t, k] holds x[t]).
    ref = orc.layout(inp["ids"], w_.N, E, w_.R)
    cnt, off = ref["cnt"], ref["expert_offset"]
    T, K = inp["ids"].shape
    src = np.full(w_.R * ref["S"], -1, np.int64)
    valid = ref["pos"] >= 0
    src[ref["pos"][valid]] = np.repeat(np.arange(T), K).reshape(T, K)[valid]
    used = np.flatnonzero(cnt > 0)
    order = used[np.argsort(-cnt[used], kind="stable")]
    experts = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    w_np = to_np(wd.reshape(E, dout, D))
    for e in experts:
        rows = np.arange(int(off[e]), int(off[e]) + int(cnt[e]))
        y_e = to_np(ys[0][torch.from_numpy(rows).cuda()])
        x_e = inp["x"][src[rows]]
        chunks = [(a, min(len(rows), a + 128)) for a in range(0, len(rows), 128)]

        def run(c, e=e, x_e=x_e, y_e=y_e):
            a, b = c
            check_gemm(orc, y_e[a:b], x_e[a:b], w_np[e][None], np.array([b - a], np.int32),
                       np.zeros(1, np.int32))

        pool_map(run, chunks)
    for b, _ in bufs:
        b.close()
    del bufs, ys, wd
    torch.cuda.empty_cache()


def test_gemm_tile_choice_follows_rows_per_expert(monkeypatch):
    # Unforced, 2-SM tiles are used when the last call routed >= 512 rows per
    # expert on average (T * K >= 512 * E), single-CTA tiles otherwise.
    monkeypatch.delenv("EP_GEMM_KERNEL", raising=False)
    D, E, K, R = 128, 4, 2, 1
    w = to_dev(W.hidden(84, E * 256, D, "bf16").reshape(E, 256, D))
    buf = ep.Buffer(1024, D, E, R, K, dtype=torch.bfloat16)
    for T, want in ((1024, 2), (1023, 1)):
        ids, sc = W.routing(85, T, E, K, "uniform", "sigmoid_norm")
        d = buf.dispatch(to_dev(W.hidden(86, T, D, "bf16")), to_dev(sc), to_dev(ids), T)
        buf.expert_gemm(d.recv_x, w)
        torch.cuda.synchronize()
        assert buf.info()["gemm_kernel"] == want, T
    assert buf.device_error() == 0
    buf.close()


def test_gemm_output_feeds_combine(orc):
    # layout -> dispatch -> expert GEMM (D -> D) -> combine on the device, as the
    # worst-token page's graph test chains them; combine of the GEMM's output is
    # bit-exact against the oracle's combine of the same rows.
    T, N, D, E, K, R = 400, 400, 256, 16, 4, 4
    x = W.hidden(80, T, D, "bf16")
    ids, sc = W.routing(80, T, E, K, "zipf", "sigmoid_norm")
    w = W.hidden(81, E * D, D, "bf16").reshape(E, D, D)
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16)
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    y = buf.expert_gemm(d.recv_x, to_dev(w))
    out = buf.combine(y, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    y_np = to_np(y.reshape(-1, D))
    want, _ = orc.combine(y_np, sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    buf.close()


@pytest.mark.parametrize("dout,kind", [(128, "1"), (512, "2"), (512, "1")])
def test_gemm_graph_replay_fresh_routing(orc, monkeypatch, dout, kind):
    # Captured once; each replay's tile list follows that replay's counts.
    monkeypatch.setenv("EP_GEMM_KERNEL", kind)
    T, N, D, E, K, R = 256, 256, 128, 8, 2, 2
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16)
    x = W.hidden(90, T, D, "bf16")
    w = W.hidden(91, E * dout, D, "bf16").reshape(E, dout, D)
    xd, wd = to_dev(x), to_dev(w)
    ids_d = torch.empty((T, K), dtype=torch.int32, device="cuda")
    sc_d = torch.empty((T, K), dtype=torch.float32, device="cuda")
    S = ep.ep_pad_tokens(N) * K
    y = torch.empty((R * S, dout), dtype=torch.bfloat16, device="cuda")
    ids0, sc0 = W.routing(92, T, E, K, "zipf", "sigmoid_norm")
    ids_d.copy_(torch.from_numpy(ids0))
    sc_d.copy_(torch.from_numpy(sc0))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d = buf.dispatch(xd, sc_d, ids_d, N, stream=s)
        buf.expert_gemm(d.recv_x, wd, y_recv=y, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        d = buf.dispatch(xd, sc_d, ids_d, N, stream=s)
        buf.expert_gemm(d.recv_x, wd, y_recv=y, stream=s)
    for i in range(4):
        ids_i, sc_i = W.routing(93 + i, T, E, K, "zipf" if i % 2 else "uniform", "sigmoid_norm")
        ids_d.copy_(torch.from_numpy(ids_i))
        sc_d.copy_(torch.from_numpy(sc_i))
        y.view(torch.int16).fill_(SENTINEL)
        g.replay()
        torch.cuda.synchronize()
        ref = orc.dispatch(x, sc_i, ids_i, N, E, R)
        check_gemm(orc, to_np(y), ref["recv_x"], w, ref["cnt"], ref["expert_offset"])
    assert buf.device_error() == 0
    buf.close()
