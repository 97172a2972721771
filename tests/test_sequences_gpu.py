"""Call sequences and concurrency against the oracle.

- Random sequences of calls on one buffer: each episode draws T <= N <= N_max,
  routing (uniform or Zipf, some pairs routed nowhere) and one way in (dispatch;
  layout then permute; per-rank dedupe then the receiver's expansion), followed
  by the calls that read the episode's layout (combine, the backward, the expert
  GEMM). Every output is compared with the oracle, so state carried from one
  call to the next (the last layout, its stride, the dedupe flag) must be right
  whatever came before.
- Two buffers driven on two streams at once, with no synchronisation between
  them: each one's outputs must equal the oracle's, as if it ran alone.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal, bits,
                      to_dev, to_np, torch_dtype)
from test_expert_gemm_gpu import SENTINEL, check_gemm

pytestmark = pytest.mark.gpu

N_MAX, D, E, K, R = 300, 128, 32, 4, 4


def episode_inputs(rng, seed, dtype):
    T = int(rng.integers(1, N_MAX + 1))
    N = int(rng.integers(T, N_MAX + 1))
    kind = "zipf" if rng.random() < 0.5 else "uniform"
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, kind, "sigmoid_norm")
    ids = ids.copy()
    drop = rng.random(ids.shape) < 0.05
    ids[drop] = -1
    return T, N, x, ids, sc


@pytest.mark.parametrize("layout", ["strided", "packed"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_call_sequences(orc, seed, layout):
    rng = np.random.default_rng(1000 + seed)
    dtype = "bf16"
    packed = layout == "packed"
    buf = ep.Buffer(N_MAX, D, E, R, K, dtype=torch_dtype(dtype), layout=layout)
    wts = W.hidden(2000 + seed, E * D, D, "bf16").reshape(E, D, D)
    wd = to_dev(wts)
    ways = ["dispatch", "layout_permute"] + ([] if packed else ["dedup"])
    for ep_i in range(12):
        T, N, x, ids, sc = episode_inputs(rng, 3000 + 100 * seed + ep_i, dtype)
        xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
        way = ways[int(rng.integers(len(ways)))]
        ref = orc.dispatch(x, sc, ids, N, E, R, packed=packed)
        S = ref["S"]
        if way == "dispatch":
            d = buf.dispatch(xd, scd, idd, N)
            y = d.recv_x
        elif way == "layout_permute":
            lay = buf.dispatch_layout(idd, N)
            d = buf.dispatch_permute(xd, scd)
            assert_layout_equal(lay, ref)
            y = d.recv_x
        else:
            dd = buf.dispatch_dedup(xd, scd, idd, N)
            y = buf.dedup_expand(idd)
            d = None
        out = buf.combine(y, scd)
        torch.cuda.synchronize()
        assert buf.device_error() == 0, (ep_i, way)
        if d is not None:
            assert_layout_equal(d.layout, ref)
            assert_recv_equal(d, ref, R)
        else:
            assert_layout_equal(dd.layout, ref)
            valid = ref["pos"][ref["pos"] >= 0]
            assert np.array_equal(bits(to_np(y.reshape(-1, D))[valid]), bits(ref["recv_x"][valid]))
        want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], S, R,
                              packed=packed)
        assert_combine_equal(to_np(out), want)
        if way == "dedup":
            continue
        follow = rng.random()
        if follow < 0.4:
            g = W.hidden(4000 + ep_i, T, D, dtype)
            grad_y, _ = buf.combine_backward(to_dev(g), y, scd, want_scores=False)
            grad_x, _ = buf.dispatch_backward(grad_y, T)
            torch.cuda.synchronize()
            assert buf.device_error() == 0
            gy_ref, _, _ = orc.combine_backward(g, ref["recv_x"], sc, ref["pos"],
                                                ref["rank_prefix"], S, R, packed=packed)
            valid = ref["pos"][ref["pos"] >= 0]
            assert np.array_equal(bits(to_np(grad_y.reshape(-1, D))[valid]), bits(gy_ref[valid]))
            gx_ref, _, _ = orc.dispatch_backward(gy_ref, None, ref["pos"], ref["rank_prefix"], S,
                                                 R, packed=packed)
            assert np.array_equal(bits(to_np(grad_x)), bits(gx_ref))
        elif follow < 0.7:
            rows = y.reshape(-1, D).shape[0]
            yg = torch.full((rows, D), SENTINEL, dtype=torch.int16, device="cuda")
            yg = yg.view(torch.bfloat16)
            buf.expert_gemm(y.reshape(rows, D), wd, y_recv=yg)
            torch.cuda.synchronize()
            assert buf.device_error() == 0
            check_gemm(orc, to_np(yg), ref["recv_x"], wts, ref["cnt"], ref["expert_offset"])
    buf.close()


def test_two_buffers_two_streams(orc):
    cfgs = [
        # (N_max, D, dtype, E, K, R, layout)
        (1000, 256, "bf16", 64, 8, 8, "strided"),
        (700, 128, "f32", 16, 2, 2, "packed"),
    ]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs, inputs = [], []
    for b, (n_max, d_, dt, e_, k_, r_, lay) in enumerate(cfgs):
        bufs.append(ep.Buffer(n_max, d_, e_, r_, k_, dtype=torch_dtype(dt), layout=lay))
        per = []
        for i in range(3):
            T = n_max - 37 * i - b
            x = W.hidden(700 + 10 * b + i, T, d_, dt)
            ids, sc = W.routing(700 + 10 * b + i, T, e_, k_, "zipf", "sigmoid_norm")
            per.append((T, x, ids, sc, to_dev(x), to_dev(ids), to_dev(sc)))
        inputs.append(per)
    torch.cuda.synchronize()
    results = [[None] * 3 for _ in cfgs]
    for i in range(3):
        for b, buf in enumerate(bufs):
            T, _, _, _, xd, idd, scd = inputs[b][i]
            s = streams[b]
            with torch.cuda.stream(s):
                out = torch.empty((T, cfgs[b][1]), dtype=buf.dtype, device="cuda")
                d = buf.dispatch(xd, scd, idd, T, stream=s)
                buf.combine(d.recv_x, scd, out=out, stream=s)
                results[b][i] = out
    torch.cuda.synchronize()
    for b, buf in enumerate(bufs):
        assert buf.device_error() == 0
        n_max, d_, dt, e_, k_, r_, lay = cfgs[b]
        for i in range(3):
            T, x, ids, sc = inputs[b][i][:4]
            ref = orc.dispatch(x, sc, ids, T, e_, r_, packed=(lay == "packed"))
            want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"],
                                  r_, packed=(lay == "packed"))
            assert_combine_equal(to_np(results[b][i]), want)
        buf.close()
