"""Backward of combine and dispatch on the GPU against the oracle.

grad_y (scattered s * grad_out) and grad_x (gather-sum in ascending k) are
compared bit for bit; the gathered receive-score gradients too. grad_scores is
a length-D dot product whose fp32 summation order is free: the oracle sums in
fp64 and rounds once, and the GPU result must lie within the classic bound for
fp32 summation, |gpu - oracle| <= (D + 2) * 2^-24 * sum_d |g_d * y_d|.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import bits, oracle_backward_all, to_dev, to_np, torch_dtype, valid_rows

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def f32_of(a):
    return (a.astype(np.uint32) << 16).view(np.float32) if a.dtype == np.uint16 else a


def assert_scores_within_bound(got, want, g, y, pos):
    """got/want [T, K]; bound from the magnitudes of the terms of each dot."""
    T, K = pos.shape
    gf = f32_of(g).astype(np.float64)
    yf = f32_of(y).astype(np.float64)
    D = gf.shape[1]
    for t in range(T):
        for k in range(K):
            p = pos[t, k]
            if p < 0:
                assert got[t, k] == 0.0
                continue
            mag = float(np.abs(gf[t] * yf[p]).sum())
            tol = (D + 2) * U * mag + 1e-37
            assert abs(float(got[t, k]) - float(want[t, k])) <= tol, (t, k, got[t, k], want[t, k])


CASES = {
    "tiny_f32":     (0xE9D15000, 13, 16, 32, 64, "f32", 8, 2, 2, "uniform", "softmax_all"),
    "ds_small":     (41, 700, 703, 704, 256, "bf16", 256, 8, 8, "zipf", "sigmoid_norm"),
    "mix_small":    (42, 1500, 1500, 1500, 512, "bf16", 8, 2, 1, "uniform", "softmax_topk"),
    "k3_f32":       (43, 333, 336, 336, 96, "f32", 48, 3, 4, "uniform", "sigmoid_norm"),
    "k16":          (44, 150, 152, 152, 128, "bf16", 64, 16, 2, "zipf", "sigmoid_norm"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_parity(orc, case):
    seed, T, N, N_max, D, dtype, E, K, R, ik, sk = CASES[case]
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, ik, sk)
    ids = ids.copy()
    if T > 5:
        ids[5, 0] = -1                        # a pair routed nowhere
    g = W.hidden(seed + 1, T, D, dtype)       # upstream gradient of out
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype))
    xd, idd, scd, gd = to_dev(x), to_dev(ids), to_dev(sc), to_dev(g)
    d = buf.dispatch(xd, scd, idd, N)
    y = d.recv_x                              # identity expert
    grad_y, gs = buf.combine_backward(gd, y, scd)
    S = d.layout.rank_stride
    h = W.normal(seed + 2, 1, R * S).astype(np.float32)   # gradient of recv_scores
    grad_x, gs_recv = buf.dispatch_backward(grad_y, T, grad_recv_scores=to_dev(h))
    torch.cuda.synchronize()
    assert buf.device_error() == 0

    ref = orc.dispatch(x, sc, ids, N, E, R)
    gy_ref, gs_ref, err = orc.combine_backward(g, ref["recv_x"], sc, ref["pos"],
                                               ref["rank_prefix"], ref["S"], R)
    assert err == 0
    pos = ref["pos"]
    valid = pos[pos >= 0]
    gy_got = to_np(grad_y.reshape(R * S, D))
    assert np.array_equal(bits(gy_got[valid]), bits(gy_ref[valid])), "grad_y differs"
    assert_scores_within_bound(to_np(gs), gs_ref, g, ref["recv_x"], pos)
    gx_ref, gsr_ref, _ = orc.dispatch_backward(gy_ref, h, pos, ref["rank_prefix"], ref["S"], R)
    assert np.array_equal(bits(to_np(grad_x)), bits(gx_ref)), "grad_x differs"
    assert np.array_equal(to_np(gs_recv).view(np.uint32), gsr_ref.view(np.uint32))
    # grad_x in fp32 before the cast
    gx32, _ = buf.dispatch_backward(grad_y, T, out_dtype=torch.float32)
    gx32_ref, _, _ = orc.dispatch_backward(gy_ref, None, pos, ref["rank_prefix"], ref["S"], R,
                                           "f32")
    assert np.array_equal(to_np(gx32).view(np.uint32), gx32_ref.view(np.uint32))
    buf.close()


def test_backward_unequal_count_runs_match():
    # [align] "Testing": forward AND backward of an unequal/unaligned run
    # reproduce the equal-count run bit for bit.
    D, E, K, R = 256, 16, 4, 4
    for a, b in [(8, 3), (6, 6), (5, 3), (13, 7)]:
        T = b
        x = W.hidden(500 + T, T, D, "bf16")
        ids, sc = W.routing(500 + T, T, E, K, "uniform", "sigmoid_norm")
        g = W.hidden(600 + T, T, D, "bf16")
        outs = []
        for N in (T, max(a, b)):
            buf = ep.Buffer(16, D, E, R, K, dtype=torch.bfloat16)
            xd, idd, scd, gd = to_dev(x), to_dev(ids), to_dev(sc), to_dev(g)
            d = buf.dispatch(xd, scd, idd, N)
            out = buf.combine(d.recv_x, scd)
            grad_y, gs = buf.combine_backward(gd, d.recv_x, scd)
            gx, _ = buf.dispatch_backward(grad_y, T)
            torch.cuda.synchronize()
            outs.append((to_np(out), to_np(gs), to_np(gx)))
            buf.close()
        for i in range(3):
            assert np.array_equal(bits(outs[0][i]), bits(outs[1][i]))


def test_backward_fullsize_deepseek(orc):
    # DeepSeek shape at full size, every element against the oracle: grad_y at
    # every valid pair and grad_x of every token bit for bit, every score
    # gradient within the fp32 summation bound (identity expert: y[pos[t,k]] =
    # x[t], so the bound's magnitudes are sum_d |g[t,d] x[t,d]|).
    w = W.WORKLOADS["deepseek"]
    inp = W.make("deepseek")
    T, D, K = w.T, w.D, w.K
    x, sc = inp["x"], inp["scores"]
    g = W.hidden(w.seed + 9, T, D, "bf16")
    buf = ep.Buffer(w.N_max, D, w.E, w.R, K, dtype=torch.bfloat16)
    xd, idd, scd, gd = to_dev(x), to_dev(inp["ids"]), to_dev(sc), to_dev(g)
    d = buf.dispatch(xd, scd, idd, w.N)
    grad_y, gs = buf.combine_backward(gd, d.recv_x, scd)
    grad_x, _ = buf.dispatch_backward(grad_y, T)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.layout(inp["ids"], w.N, w.E, w.R)
    pos = ref["pos"]
    assert np.array_equal(to_np(d.layout.pos), pos)
    gy_ref, gs_ref, gx_ref = oracle_backward_all(orc, x, g, sc, pos)
    assert np.array_equal(valid_rows(grad_y, pos), gy_ref), "grad_y differs from the oracle"
    assert np.array_equal(to_np(grad_x), gx_ref), "grad_x differs from the oracle"
    mag = np.abs(f32_of(g).astype(np.float64) * f32_of(x).astype(np.float64)).sum(1)
    tol = (D + 2) * U * mag[:, None] + 1e-37
    got = to_np(gs).astype(np.float64)
    assert np.all(got[pos < 0] == 0.0)
    bad = (np.abs(got - gs_ref.astype(np.float64)) > tol) & (pos >= 0)
    assert not bad.any(), f"{int(bad.sum())} score gradients outside the bound"
    buf.close()
    torch.cuda.empty_cache()
