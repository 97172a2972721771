"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Oracle-sized cases compare everything: layout arrays, every defined receive
row with its score and source, and the combine output (bf16 bit-exact; fp32
before the cast bit-exact, which is inside the 1e-6 relative allowance).
Cases span several layout tiles with a ragged last tile, non-multiple-of-4
token counts, N > T padding, empty calls, odd K, fp32 rows, bad and
duplicated ids, and both permute implementations.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import (assert_combine_equal, assert_layout_equal, assert_recv_equal, bits,
                      to_dev, to_np, torch_dtype)

pytestmark = pytest.mark.gpu

# vec: 16-byte vector permute; bulk: the default bulk dispatch (one cooperative
# kernel: counts, grid barrier, prefix, positions, copies; calls of up to 4096
# pairs count every id in every CTA instead of meeting at the barrier);
# bulk_barrier: the same with every call meeting at the barrier
# (EP_DISPATCH_SMALL_PAIRS=0); fused: the bulk dispatch as count + scan + fused
# positions/copy kernels (EP_DISPATCH_ONEPASS=0)
IMPLS = ["vec", "bulk", "bulk_barrier", "fused"]
IMPL_IDS = IMPLS


@pytest.fixture
def impl(request, monkeypatch):
    if request.param == "fused":
        monkeypatch.setenv("EP_DISPATCH_ONEPASS", "0")
    if request.param == "bulk_barrier":
        monkeypatch.setenv("EP_DISPATCH_SMALL_PAIRS", "0")
    return ep.EP_PERMUTE_VEC if request.param == "vec" else ep.EP_PERMUTE_BULK

# id: (seed, T, N, N_max, D, dtype, E, K, R, ids, scores)
CASES = {
    "tiny":             (0xE9D15000, 16, 16, 32, 64, "f32", 8, 2, 2, "uniform", "softmax_all"),
    "tiny_N32":         (0xE9D15000, 16, 32, 32, 64, "f32", 8, 2, 2, "uniform", "softmax_all"),
    "tiny_T13_N16":     (0xE9D15000, 13, 16, 32, 64, "f32", 8, 2, 2, "uniform", "softmax_all"),
    "tiny_T1":          (7, 1, 1, 32, 64, "f32", 8, 2, 2, "uniform", "softmax_all"),
    "tiny_bf16":        (8, 29, 31, 32, 64, "bf16", 8, 2, 2, "uniform", "softmax_all"),
    "ds_small_tiles":   (9, 1000, 1003, 1024, 256, "bf16", 256, 8, 8, "zipf", "sigmoid_norm"),
    "mix_small_tiles":  (10, 3001, 3001, 4096, 512, "bf16", 8, 2, 1, "uniform", "softmax_topk"),
    "k3_e48_r4_f32":    (11, 777, 800, 800, 96, "f32", 48, 3, 4, "uniform", "sigmoid_norm"),
    "k1_e4_r4":         (12, 2049, 2049, 2050, 64, "bf16", 4, 1, 4, "uniform", "sigmoid_norm"),
    "k16_e64_r2":       (13, 300, 301, 512, 128, "bf16", 64, 16, 2, "zipf", "sigmoid_norm"),
    "k40_e64_r8":       (14, 90, 90, 96, 64, "bf16", 64, 40, 8, "uniform", "sigmoid_norm"),
    "e1024_r64":        (15, 700, 702, 702, 32, "bf16", 1024, 8, 64, "uniform", "sigmoid_norm"),
}


def case_inputs(seed, T, D, dtype, E, K, ids_kind, scores_kind):
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, ids_kind, scores_kind)
    return x, ids, sc


def run_and_check(orc, x, ids, sc, N, N_max, D, dtype, E, K, R, impl):
    T = ids.shape[0]
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=impl)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, N)
    out = buf.combine(d.recv_x, scd)
    out32 = buf.combine(d.recv_x, scd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert buf.device_error() == ref["err"]
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    want32, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R, "f32")
    assert_combine_equal(to_np(out32), want32)
    buf.close()


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS, indirect=True)
@pytest.mark.parametrize("case", sorted(CASES))
def test_parity(orc, case, impl):
    seed, T, N, N_max, D, dtype, E, K, R, ik, sk = CASES[case]
    x, ids, sc = case_inputs(seed, T, D, dtype, E, K, ik, sk)
    run_and_check(orc, x, ids, sc, N, N_max, D, dtype, E, K, R, impl)


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS, indirect=True)
def test_empty_calls(orc, impl):
    D, E, K, R = 64, 8, 2, 2
    buf = ep.Buffer(32, D, E, R, K, dtype=torch.float32, permute_impl=impl)
    for N in (0, 5):
        x = torch.empty((0, D), dtype=torch.float32, device="cuda")
        ids = torch.empty((0, K), dtype=torch.int32, device="cuda")
        sc = torch.empty((0, K), dtype=torch.float32, device="cuda")
        d = buf.dispatch(x, sc, ids, N)
        out = buf.combine(d.recv_x, sc)
        torch.cuda.synchronize()
        ref = orc.layout(np.zeros((0, K), np.int32), N, E, R)
        assert_layout_equal(d.layout, ref)
        assert out.shape == (0, D)
    assert buf.device_error() == 0


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS, indirect=True)
def test_bad_and_duplicate_ids(orc, impl):
    # -1 routes nowhere; ids outside [-1, E) are treated as -1 and reported;
    # a repeated id gets one row per occurrence.
    T, N, D, E, K, R = 37, 40, 64, 16, 4, 4
    x, ids, sc = case_inputs(21, T, D, "bf16", E, K, "uniform", "sigmoid_norm")
    ids = ids.copy()
    ids[0] = [3, 3, 3, 3]
    ids[1, 2] = -1
    ids[5, 0] = E
    ids[6, 3] = -7
    ids[36] = [-1, -1, -1, -1]
    buf = ep.Buffer(64, D, E, R, K, dtype=torch.bfloat16, permute_impl=impl)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, N)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert ref["err"] & 1
    assert buf.device_error() & ep.EP_DEVERR_BAD_ID
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    got = to_np(out)
    assert_combine_equal(got, want)
    assert not got[36].any()                 # a token with no expert combines to +0


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS, indirect=True)
def test_scaled_experts(orc, impl):
    # Expert stand-in y = 2^((e mod 4) - 1) * recv_x (exact in bf16) between
    # dispatch and combine: a wrong row or k in the gather changes the result.
    T, N, D, E, K, R = 513, 516, 256, 32, 4, 4
    x, ids, sc = case_inputs(22, T, D, "bf16", E, K, "zipf", "sigmoid_norm")
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16, permute_impl=impl)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, N)
    src = d.recv_src.reshape(-1).clamp(0, T * K - 1).long()
    e_row = idd.reshape(-1).long()[src]
    scale = torch.exp2(((e_row % 4) - 1).float())
    y = (d.recv_x.reshape(-1, D).float() * scale[:, None]).to(torch.bfloat16)
    out = buf.combine(y, scd)
    torch.cuda.synchronize()
    ref = orc.dispatch(x, sc, ids, N, E, R)
    yref = ref["recv_x"].copy()
    for t in range(T):
        for k in range(K):
            p = ref["pos"][t, k]
            v = (yref[p].astype(np.uint32) << 16).view(np.float32) * np.float32(
                2.0 ** ((ids[t, k] % 4) - 1))
            yref[p] = (v.view(np.uint32) >> 16).astype(np.uint16)
    want, _ = orc.combine(yref, sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)


def test_unequal_count_runs_match(orc):
    # A token's combined output depends only on its own routing: the same
    # tokens dispatched at their own padded count and at a larger group max
    # give identical bits (combos from the pages' functional test).
    D, E, K, R = 128, 16, 4, 4
    for a, b in [(8, 3), (6, 6), (5, 3), (13, 7)]:
        group = max(a, b)
        for T in (a, b):
            x, ids, sc = case_inputs(100 + T, T, D, "bf16", E, K, "uniform", "sigmoid_norm")
            outs = []
            for N in (T, group):
                buf = ep.Buffer(16, D, E, R, K, dtype=torch.bfloat16)
                xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
                d = buf.dispatch(xd, scd, idd, N)
                outs.append(to_np(buf.combine(d.recv_x, scd)))
                assert d.layout.padded_tokens == ((N + 3) // 4) * 4
            assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("impl", IMPLS, ids=IMPL_IDS, indirect=True)
@pytest.mark.parametrize("case", ["tiny_T13_N16", "ds_small_tiles", "k3_e48_r4_f32",
                                  "k40_e64_r8", "e1024_r64"])
def test_parity_packed_layout(orc, case, impl):
    # Exact-mode layout: ranks back to back, valid rows exactly [0, true total);
    # forward and backward against the oracle's packed definition.
    seed, T, N, N_max, D, dtype, E, K, R, ik, sk = CASES[case]
    x, ids, sc = case_inputs(seed, T, D, dtype, E, K, ik, sk)
    g = W.hidden(seed + 5, T, D, dtype)
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=impl,
                    layout="packed")
    xd, idd, scd, gd = to_dev(x), to_dev(ids), to_dev(sc), to_dev(g)
    d = buf.dispatch(xd, scd, idd, N)
    out = buf.combine(d.recv_x, scd)
    grad_y, _ = buf.combine_backward(gd, d.recv_x, scd, want_scores=False)
    grad_x, _ = buf.dispatch_backward(grad_y, T)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R, packed=True)
    assert d.layout.packed
    assert_layout_equal(d.layout, ref)
    total = int(ref["rank_prefix"][-1])
    assert np.array_equal(bits(to_np(d.recv_x)[:total]), bits(ref["recv_x"][:total]))
    assert np.array_equal(to_np(d.recv_src)[:total], ref["recv_src"][:total])
    assert np.array_equal(to_np(d.recv_scores)[:total].view(np.uint32),
                          ref["recv_scores"][:total].view(np.uint32))
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R,
                          packed=True)
    assert_combine_equal(to_np(out), want)
    gy_ref, _, _ = orc.combine_backward(g, ref["recv_x"], sc, ref["pos"], ref["rank_prefix"],
                                        ref["S"], R, packed=True)
    assert np.array_equal(bits(to_np(grad_y)[:total]), bits(gy_ref[:total]))
    gx_ref, _, _ = orc.dispatch_backward(gy_ref, None, ref["pos"], ref["rank_prefix"], ref["S"],
                                         R, packed=True)
    assert np.array_equal(bits(to_np(grad_x)), bits(gx_ref))
    buf.close()


@pytest.mark.parametrize("onepass,launches", [("1", 1), ("0", 3)])
def test_bulk_dispatch_launch_count(orc, monkeypatch, onepass, launches):
    # The default bulk dispatch is one cooperative kernel; without it, count,
    # scan and the fused positions/copy kernel. Both match the oracle.
    monkeypatch.setenv("EP_DISPATCH_ONEPASS", onepass)
    seed, T, N, N_max, D, dtype, E, K, R, ik, sk = CASES["ds_small_tiles"]
    x, ids, sc = case_inputs(seed, T, D, dtype, E, K, ik, sk)
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype))
    n0 = buf.info()["kernel_launches"]
    d = buf.dispatch(to_dev(x), to_dev(sc), to_dev(ids), N)
    torch.cuda.synchronize()
    assert buf.info()["kernel_launches"] - n0 == launches
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    # back-to-back calls reuse the grid barrier; a later call still matches
    ids2, sc2 = W.routing(seed + 1, T, E, K, "uniform", sk)
    for _ in range(3):
        d = buf.dispatch(to_dev(x), to_dev(sc2), to_dev(ids2), N)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref2 = orc.dispatch(x, sc2, ids2, N, E, R)
    assert_layout_equal(d.layout, ref2)
    assert_recv_equal(d, ref2, R)
    buf.close()
