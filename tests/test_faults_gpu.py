"""Failure detection without faulting the GPU.

Host-side argument errors return a status and enqueue nothing (no kernel
launch is counted). Data errors found on the device set sticky bits in the
buffer's error word and never lead to an out-of-bounds access: the inputs
here are crafted so the kernels' own checks turn them into errors (bad ids,
a receive row past its rank's true total). Synchronous calls refuse to run
while the stream is capturing.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
from combine_topk_ids_expert_gb300 import _abi
import workloads as W
from gpu_util import assert_combine_equal, to_dev, to_np

pytestmark = pytest.mark.gpu

D, E, K, R = 64, 16, 4, 4


def small(T=21, seed=3, dtype="bf16"):
    x = W.hidden(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, "uniform", "sigmoid_norm")
    return x, ids, sc


def launches(buf):
    return buf.info()["kernel_launches"]


def test_argument_errors_enqueue_nothing():
    buf = ep.Buffer(32, D, E, R, K, dtype=torch.bfloat16)
    x, ids, sc = small()
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    h = buf.handle
    n0 = launches(buf)
    cases = [
        (lambda: ep.ep_dispatch(h, xd, scd, idd, 21, 20), _abi.EP_ERR_INVALID_ARG),   # T > N
        (lambda: ep.ep_dispatch(h, xd, scd, idd, 21, 33), _abi.EP_ERR_CAPACITY),      # N > N_max
        (lambda: ep.ep_dispatch(h, xd, scd, idd, -1, 4), _abi.EP_ERR_INVALID_ARG),
        (lambda: ep.ep_combine(h, xd, scd, 21, xd, 0), _abi.EP_ERR_NO_LAYOUT),       # no layout yet
        (lambda: ep.ep_dispatch_permute(h, xd, scd), _abi.EP_ERR_NO_LAYOUT),
        (lambda: ep.ep_dispatch_layout(h, idd, 21, 40), _abi.EP_ERR_CAPACITY),
    ]
    for call, want in cases:
        with pytest.raises(ep.EpError) as ei:
            call()
        assert ei.value.status == want
    # misaligned hidden rows: a view starting 2 bytes into a tensor
    big = torch.zeros(21 * D + 1, dtype=torch.bfloat16, device="cuda")
    mis = big[1:].view(21, D)
    with pytest.raises(ep.EpError) as ei:
        ep.ep_dispatch(h, mis, scd, idd, 21, 21)
    assert ei.value.status == _abi.EP_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert launches(buf) == n0
    # after a valid dispatch, combine with another T is refused
    buf.dispatch(xd, scd, idd, 24)
    n1 = launches(buf)
    with pytest.raises(ep.EpError) as ei:
        ep.ep_combine(h, xd, scd[:20].contiguous(), 20, xd, 0)
    assert ei.value.status == _abi.EP_ERR_NO_LAYOUT
    with pytest.raises(ep.EpError) as ei:
        ep.ep_combine(h, xd, scd, 21, mis, 0)
    assert ei.value.status == _abi.EP_ERR_ALIGNMENT
    with pytest.raises(ep.EpError) as ei:
        ep.ep_combine(h, xd, scd, 21, xd, 7)
    assert ei.value.status == _abi.EP_ERR_INVALID_ARG
    assert launches(buf) == n1
    assert buf.device_error() == 0
    buf.close()


def test_workspace_checks():
    cfg = _abi.EpConfig(32, D, E, R, K, _abi.EP_BF16, 0, 0)
    n = ep.ep_buffer_required_bytes(cfg)
    small_ws = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ep.EpError) as ei:
        ep.ep_buffer_init(cfg, small_ws)
    assert ei.value.status == _abi.EP_ERR_WORKSPACE
    ws = torch.empty(n + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(ep.EpError) as ei:
        ep.ep_buffer_init(cfg, ws[16:])                # not 256-byte aligned
    assert ei.value.status == _abi.EP_ERR_WORKSPACE
    import ctypes as C
    host = torch.empty(n, dtype=torch.uint8).pin_memory()
    hh = C.c_void_p()
    st = _abi.lib().ep_buffer_init(C.byref(cfg), host.data_ptr(), n, C.byref(hh))
    assert st == _abi.EP_ERR_WORKSPACE                  # host memory is not a device workspace
    h = ep.ep_buffer_init(cfg, ws[:n])
    ep.ep_buffer_destroy(h)


def test_synchronous_calls_refused_while_capturing():
    buf = ep.Buffer(32, D, E, R, K, dtype=torch.bfloat16)
    x, ids, sc = small()
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    buf.dispatch(xd, scd, idd, 24)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    errs = []
    with torch.cuda.graph(g, stream=s):
        for call in (lambda: buf.dispatch_layout(idd, 24, stream=s, host_counts=True),
                     lambda: buf.device_error(stream=s)):
            try:
                call()
            except ep.EpError as e:
                errs.append(e.status)
        buf.dispatch(xd, scd, idd, 24, stream=s)       # the asynchronous path captures fine
    assert errs == [_abi.EP_ERR_CAPTURE_HOST_SYNC] * 2
    g.replay()
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    buf.close()


def test_exact_mode_host_counts(orc):
    buf = ep.Buffer(32, D, E, R, K, dtype=torch.bfloat16)
    x, ids, sc = small(T=29, seed=5)
    lay, host = buf.dispatch_layout(to_dev(ids), 31, host_counts=True)
    ref = orc.layout(ids, 31, E, R)
    assert np.array_equal(host.numpy(), ref["cnt"])
    assert np.array_equal(to_np(lay.tokens_per_expert), ref["cnt"])
    buf.close()


def test_row_past_true_total_is_rejected(orc):
    # Point one pair at the first row after rank 0's true total (stale data):
    # combine must skip it, report EP_DEVERR_ROW_OOB, and match the oracle,
    # which applies the same rule.
    buf = ep.Buffer(32, D, E, R, K, dtype=torch.bfloat16)
    x, ids, sc = small(T=21, seed=6)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, 24)
    torch.cuda.synchronize()
    pos = to_np(d.layout.pos).copy()
    rows0 = int(to_np(d.layout.rows_per_rank)[0])
    pos[0, 0] = rows0                       # first row past rank 0's total
    pos[1, 1] = 10 ** 8                     # far outside every rank
    d.layout.pos.copy_(torch.from_numpy(pos))
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() & ep.EP_DEVERR_ROW_OOB
    ref = orc.dispatch(x, sc, ids, 24, E, R)
    want, err = orc.combine(ref["recv_x"], sc, pos, ref["rank_prefix"], ref["S"], R)
    assert err & 2
    assert_combine_equal(to_np(out), want)
    assert buf.device_error() == 0          # cleared by the previous read
    buf.close()


def test_bad_ids_are_reported_and_contained(orc):
    buf = ep.Buffer(32, D, E, R, K, dtype=torch.bfloat16)
    x, ids, sc = small(T=16, seed=7)
    ids = ids.copy()
    ids[3, 1] = 1 << 20
    ids[4, 0] = -(1 << 20)
    d = buf.dispatch(to_dev(x), to_dev(sc), to_dev(ids), 16)
    torch.cuda.synchronize()
    assert buf.device_error() == ep.EP_DEVERR_BAD_ID
    ref = orc.layout(ids, 16, E, R)
    assert np.array_equal(to_np(d.layout.pos), ref["pos"])
    assert to_np(d.layout.pos)[3, 1] == -1 and to_np(d.layout.pos)[4, 0] == -1
    buf.close()


def test_bounded_wait_runs_out_and_reports(orc, monkeypatch):
    # The bulk permute waits on an mbarrier for each row load with a 2 s limit.
    # EP_TEST_SKIP_LOAD makes CTA 0 never issue one load, so that wait runs
    # out: the kernel must set EP_DEVERR_TIMEOUT, let its other loads land and
    # return, leaving the context usable. Nothing faults or hangs.
    monkeypatch.setenv("EP_TEST_SKIP_LOAD", "0")
    buf = ep.Buffer(64, D, E, R, K, dtype=torch.bfloat16, permute_impl=ep.EP_PERMUTE_BULK)
    monkeypatch.delenv("EP_TEST_SKIP_LOAD")
    x, ids, sc = small(T=40, seed=8)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    buf.dispatch(xd, scd, idd, 40)
    torch.cuda.synchronize()
    assert buf.device_error() & ep.EP_DEVERR_TIMEOUT
    buf.close()
    # The same GPU context keeps working: a fresh buffer is oracle-exact.
    good = ep.Buffer(64, D, E, R, K, dtype=torch.bfloat16, permute_impl=ep.EP_PERMUTE_BULK)
    d = good.dispatch(xd, scd, idd, 40)
    out = good.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert good.device_error() == 0
    ref = orc.dispatch(x, sc, ids, 40, E, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    good.close()


def test_grid_barrier_runs_out_and_recovers(orc, monkeypatch):
    # The one-pass dispatch meets all its CTAs at a grid barrier (words at the
    # end of the workspace: even-generation arrivals, generation, pool counter,
    # odd-generation arrivals) with a 2 s limit. Seeding the first arrival
    # count past the grid size means the count never equals the grid size, so
    # every CTA's wait runs out: the kernel must report
    # EP_DEVERR_TIMEOUT and return; reading the flag starts the barrier over,
    # and the next dispatch on the same buffer is oracle-exact. (A call this
    # small would skip the barrier: EP_DISPATCH_SMALL_PAIRS=0 keeps it.)
    monkeypatch.setenv("EP_DISPATCH_SMALL_PAIRS", "0")
    buf = ep.Buffer(64, D, E, R, K, dtype=torch.bfloat16, permute_impl=ep.EP_PERMUTE_BULK)
    x, ids, sc = small(T=40, seed=9)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    ws = buf.workspace
    align = 256                      # workspace carve granularity
    gbar = ws.numel() - 2 * align    # the barrier's four words, then the error word
    ws[gbar:gbar + 4].view(torch.int32).fill_(1 << 20)
    n0 = buf.info()["kernel_launches"]
    buf.dispatch(xd, scd, idd, 40)
    torch.cuda.synchronize()
    assert buf.info()["kernel_launches"] - n0 == 1, "expected the one-pass dispatch"
    assert buf.device_error() & ep.EP_DEVERR_TIMEOUT
    assert int(ws[gbar:gbar + 16].view(torch.int32).abs().sum().item()) == 0
    d = buf.dispatch(xd, scd, idd, 40)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, 40, E, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    buf.close()


def test_grid_barrier_opened_early_stays_in_bounds(orc, monkeypatch):
    # Corrupted barrier words can open the barrier before every CTA has
    # counted its tile: seeding the arrival count at three below the grid size
    # (a 40-token call runs 40 CTAs, one token each) lets the first three CTAs
    # through with the tile tables of nobody else. Their layout is garbage,
    # but every store stays inside the receive buffer (rows outside the call's
    # R * S are skipped and reported as EP_DEVERR_ROW_OOB), the other CTAs'
    # waits run out (EP_DEVERR_TIMEOUT: their count passes the grid size), and
    # after the host resets the words the next dispatch is oracle-exact.
    monkeypatch.setenv("EP_DISPATCH_SMALL_PAIRS", "0")
    buf = ep.Buffer(64, D, E, R, K, dtype=torch.bfloat16, permute_impl=ep.EP_PERMUTE_BULK)
    x, ids, sc = small(T=40, seed=11)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    ws = buf.workspace
    gbar = ws.numel() - 2 * 256      # the barrier's four words, then the error word
    ws[gbar:gbar + 4].view(torch.int32).fill_(40 - 3)
    n0 = buf.info()["kernel_launches"]
    buf.dispatch(xd, scd, idd, 40)
    torch.cuda.synchronize()
    assert buf.info()["kernel_launches"] - n0 == 1, "expected the one-pass dispatch"
    flags = buf.device_error()
    assert flags & ep.EP_DEVERR_TIMEOUT
    assert flags & ~(ep.EP_DEVERR_TIMEOUT | ep.EP_DEVERR_ROW_OOB) == 0
    assert int(ws[gbar:gbar + 16].view(torch.int32).abs().sum().item()) == 0
    d = buf.dispatch(xd, scd, idd, 40)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, 40, E, R)
    want, _ = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R)
    assert_combine_equal(to_np(out), want)
    buf.close()


def test_dedupe_grid_barrier_runs_out_and_recovers(orc):
    # The one-pass dedupe meets its CTAs at the same grid barrier as the
    # dispatch: with the arrival count seeded past the grid size every wait
    # runs out, the kernel reports EP_DEVERR_TIMEOUT after its loads land,
    # and after the host resets the words the next dedupe is oracle-exact.
    buf = ep.Buffer(64, D, E, R, K, dtype=torch.bfloat16)
    x, ids, sc = small(T=40, seed=13)
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    ws = buf.workspace
    gbar = ws.numel() - 2 * 256      # the barrier's four words, then the error word
    ws[gbar:gbar + 4].view(torch.int32).fill_(1 << 20)
    n0 = buf.info()["kernel_launches"]
    buf.dispatch_dedup(xd, scd, idd, 40)
    torch.cuda.synchronize()
    assert buf.info()["kernel_launches"] - n0 == 1, "expected the one-pass dedupe"
    assert buf.device_error() & ep.EP_DEVERR_TIMEOUT
    assert int(ws[gbar:gbar + 16].view(torch.int32).abs().sum().item()) == 0
    dd = buf.dispatch_dedup(xd, scd, idd, 40)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch_dedup(x, sc, ids, 40, E, R)
    assert np.array_equal(to_np(dd.tok_pos), ref["tok_pos"])
    assert np.array_equal(to_np(dd.layout.tokens_in_rank), ref["tokens_in_rank"])
    buf.close()
