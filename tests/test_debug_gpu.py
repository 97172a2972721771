"""Debugging aids: the receive-buffer sentinel checks (EP_DEBUG=1), NVTX ranges
(EP_NVTX=1) and the SM budget from the environment (EP_NUM_SMS).

With EP_DEBUG=1 the dispatch fills its receive rows with 0xFF, permutes, and
checks that every row inside a rank's true total was written and every row
past it was not; the combine repeats the check when it reads the receive
buffer itself. Clean runs must stay oracle-exact with no flag raised; a
planted write past a rank's total and a planted sentinel inside it must each
raise their flag (the mistakes are planted from the host, between calls).
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_combine_equal, assert_layout_equal, to_dev, to_np, torch_dtype

pytestmark = pytest.mark.gpu

CASES = {
    # name: (seed, T, N, N_max, D, dtype, E, K, R, ids, layout, impl)
    "bulk_strided": (140, 700, 703, 720, 256, "bf16", 64, 8, 8, "zipf", "strided",
                     ep.EP_PERMUTE_BULK),
    "vec_strided": (141, 300, 300, 320, 96, "f32", 16, 3, 4, "uniform", "strided",
                    ep.EP_PERMUTE_VEC),
    "bulk_packed": (142, 500, 501, 512, 128, "bf16", 32, 4, 4, "zipf", "packed",
                    ep.EP_PERMUTE_BULK),
}


def run(orc, case):
    seed, T, N, N_max, D, dtype, E, K, R, ik, layout, impl = CASES[case]
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, ik, "sigmoid_norm")
    buf = ep.Buffer(N_max, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=impl,
                    layout=layout)
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    torch.cuda.synchronize()
    ref = orc.dispatch(x, sc, ids, N, E, R, packed=(layout == "packed"))
    return buf, d, scd, ref, sc


@pytest.mark.parametrize("case", sorted(CASES))
def test_sentinel_checks_pass_on_clean_runs(orc, monkeypatch, case):
    monkeypatch.setenv("EP_DEBUG", "1")
    buf, d, scd, ref, sc = run(orc, case)
    assert buf.device_error() == 0
    assert_layout_equal(d.layout, ref)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    R = buf.R
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R,
                          packed=(buf.packed))
    assert_combine_equal(to_np(out), want)
    buf.close()


def test_sentinel_flags_a_write_past_a_ranks_total(orc, monkeypatch):
    monkeypatch.setenv("EP_DEBUG", "1")
    buf, d, scd, ref, _ = run(orc, "bulk_strided")
    assert buf.device_error() == 0
    S = ref["S"]
    r = int(np.argmin(ref["rows_per_rank"]))          # a rank with spare rows
    row = int(ref["rows_per_rank"][r])
    assert row < S
    d.recv_x.reshape(-1, S, buf.D)[r, row, :8] = 1.0   # planted between the calls
    buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() & ep.EP_DEVERR_DEBUG_STRAY
    buf.close()


def test_sentinel_flags_an_unwritten_row(orc, monkeypatch):
    monkeypatch.setenv("EP_DEBUG", "1")
    buf, d, scd, ref, _ = run(orc, "bulk_packed")
    assert buf.device_error() == 0
    flat = d.recv_x.reshape(-1, buf.D).view(torch.int16)
    flat[3, :8] = -1                                    # 0xFFFF: the sentinel bytes
    buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() & ep.EP_DEVERR_DEBUG_UNWRITTEN
    buf.close()


def test_num_sms_and_nvtx_from_the_environment(orc, monkeypatch):
    monkeypatch.setenv("EP_NUM_SMS", "40")
    monkeypatch.setenv("EP_NVTX", "1")
    buf, d, scd, ref, sc = run(orc, "bulk_strided")
    assert buf.info()["num_sms"] == 40
    assert buf.device_error() == 0
    assert_layout_equal(d.layout, ref)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], buf.R)
    assert_combine_equal(to_np(out), want)
    buf.close()
