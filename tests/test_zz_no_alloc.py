"""ep_dispatch_layout_noalloc: the dispatch layout for callers that cannot
allocate device memory (for example an op inside a host framework that owns
every device allocation and only hands it input and output tensors). It takes
the ids and caller-owned outputs and uses a fixed library-owned device array
for its tile tables, so it never allocates.

Its results must equal the oracle's layout (and those of the buffer-based
ep_dispatch_layout) bit for bit. This file is named to be collected last, so a
failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W

FIELDS = (("cnt", "tokens_per_expert"), ("expert_offset", "expert_offset"),
          ("rows_per_rank", "rows_per_rank"), ("rank_prefix", "rank_prefix"),
          ("tokens_in_rank", "tokens_in_rank"), ("pos", "pos"))


def poisoned_outputs(T, K, E, R):
    def full(*shape):
        return torch.full(shape, -7, dtype=torch.int32, device="cuda")
    return {"tokens_per_expert": full(E), "expert_offset": full(E), "rows_per_rank": full(R),
            "rank_prefix": full(R), "tokens_in_rank": full(R), "pos": full(T, K)}


def spread_ids(seed, T, E, K):
    """Ids drawn uniformly with replacement (a token may pick an expert twice,
    which the layout allows): a fast generator for the large cases."""
    return (W.u64(seed, 77, T * K) % np.uint64(E)).astype(np.int32).reshape(T, K)


def run_noalloc(ids_np, N, K, E, R, with_flags=True):
    T = ids_np.shape[0]
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).cuda().reshape(T, K)
    out = poisoned_outputs(T, K, E, R)
    err = torch.zeros(1, dtype=torch.int32, device="cuda") if with_flags else None
    ep.ep_dispatch_layout_noalloc(ids, T, N, K, E, R, **out, error_flags=err)
    torch.cuda.synchronize()
    return out, (None if err is None else int(err.item()))


def assert_equals_oracle(orc, out, ids_np, N, E, R):
    ref = orc.layout(ids_np, N, E, R)
    for rname, name in FIELDS:
        got = out[name].cpu().numpy()
        assert np.array_equal(got.reshape(ref[rname].shape), ref[rname]), name
    return ref


def test_scratch_bound_is_host_arithmetic():
    # The bound the entry point enforces, from the host-only size query (no
    # device is touched): tile tables of max(1, 2048/K)-token tiles.
    cap = ep.EP_NOALLOC_SCRATCH_BYTES
    assert cap == 4 << 20
    need = ep.ep_dispatch_layout_noalloc_scratch_bytes
    assert need(516_000, 8, 256, 8) <= cap < need(600_000, 8, 256, 8)
    assert need(126_000, 8, 1024, 64) <= cap < need(130_000, 8, 1024, 64)
    assert need(0, 8, 256, 8) <= 1024
    assert need(-1, 8, 256, 8) == 0 and need(10, 0, 256, 8) == 0
    # monotone in the token count
    sizes = [need(t, 8, 256, 8) for t in range(0, 20_000, 97)]
    assert sizes == sorted(sizes)


@pytest.mark.gpu
def test_noalloc_layout_matches_buffer_layout_on_two_calls(orc):
    E, K, R = 256, 8, 8
    # Two calls in a row through the C ABI: a ragged multi-tile call with
    # padding, then the full DeepSeek-shaped routing (Zipf ids, 8192 tokens).
    calls = [(W.topk_ids_zipf(51, 1000, E, K), 1003),
             (W.topk_ids_zipf(W.WORKLOADS["deepseek"].seed, 8192, E, K), 8192)]
    buf = ep.Buffer(8192, 64, E, R, K, dtype=torch.bfloat16)
    for ids_np, N in calls:
        lay = buf.dispatch_layout(torch.from_numpy(ids_np).cuda(), N)
        out, err = run_noalloc(ids_np, N, K, E, R)
        for _, name in FIELDS:   # integer results: bit-exact, as for every layout test
            assert torch.equal(out[name], getattr(lay, name)), name
        assert_equals_oracle(orc, out, ids_np, N, E, R)
        assert err == 0
        assert buf.device_error() == 0
    buf.close()


CASES = {
    # name: (seed, T, N, E, K, R, ids)
    "tiny": (0xE9D15000, 16, 16, 8, 2, 2, "uniform"),
    "tiny_ragged": (3, 13, 16, 8, 2, 2, "uniform"),
    "mixtral": (0xE9D15001, 4096, 4096, 8, 2, 1, "uniform"),
    "empty": (4, 0, 8, 256, 8, 8, "uniform"),
    "one_token": (5, 1, 1, 256, 8, 8, "zipf"),
    "k64": (6, 700, 703, 128, 64, 4, "uniform"),
    "e1024_r64_near_limit": (7, 126_000, 126_000, 1024, 8, 64, "spread"),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_oracle(orc, case):
    seed, T, N, E, K, R, kind = CASES[case]
    gen = {"zipf": W.topk_ids_zipf, "uniform": W.topk_ids_uniform, "spread": spread_ids}[kind]
    ids_np = gen(seed, T, E, K).reshape(T, K)
    out, err = run_noalloc(ids_np, N, K, E, R)
    ref = assert_equals_oracle(orc, out, ids_np, N, E, R)
    assert err == 0 and ref["err"] == 0


@pytest.mark.gpu
@pytest.mark.parametrize("with_flags", [True, False], ids=["flags", "no_flags"])
def test_noalloc_bad_ids(orc, with_flags):
    # Ids outside [-1, E) are treated as -1 and reported as EP_DEVERR_BAD_ID in
    # the caller's word; without one, the report goes nowhere and the layout is
    # the same.
    T, N, E, K, R = 300, 302, 64, 4, 4
    ids_np = W.topk_ids_uniform(8, T, E, K).reshape(T, K).copy()
    ids_np[3, 1], ids_np[77, 0], ids_np[299, 3], ids_np[10, 2] = E, -2, 1 << 30, -1
    out, err = run_noalloc(ids_np, N, K, E, R, with_flags)
    ref = assert_equals_oracle(orc, out, ids_np, N, E, R)
    assert ref["err"] == ep.EP_DEVERR_BAD_ID
    if with_flags:
        assert err == ep.EP_DEVERR_BAD_ID


@pytest.mark.gpu
def test_noalloc_small_call_after_a_large_one(orc):
    # The shared array keeps the last call's tables; a 64-token call right after
    # a 500k-token call must not see them.
    E, K, R = 256, 8, 8
    big = spread_ids(9, 500_000, E, K)
    out, err = run_noalloc(big, 500_000, K, E, R)
    assert_equals_oracle(orc, out, big, 500_000, E, R)
    assert err == 0
    small = W.topk_ids_uniform(10, 64, E, K)
    out, err = run_noalloc(small, 66, K, E, R)
    assert_equals_oracle(orc, out, small, 66, E, R)
    assert err == 0


@pytest.mark.gpu
def test_noalloc_rejects_bad_arguments_before_launching():
    # Sizes beyond the array: EP_ERR_CAPACITY, with real tensors (nothing is
    # launched); tensors too small for the sizes: refused by the binding.
    E, K, R = 256, 8, 8
    T = 600_000
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    out = poisoned_outputs(T, K, E, R)
    with pytest.raises(ep.EpError) as e:
        ep.ep_dispatch_layout_noalloc(ids, T, T, K, E, R, **out)
    assert e.value.status == ep._abi.EP_ERR_CAPACITY
    assert int(out["tokens_per_expert"][0]) == -7          # untouched
    small = poisoned_outputs(10, K, E, R)
    ids10 = torch.zeros((10, K), dtype=torch.int32, device="cuda")
    for name, bad in (("pos", torch.zeros((9, K), dtype=torch.int32, device="cuda")),
                      ("rank_prefix", torch.zeros(R - 1, dtype=torch.int32, device="cuda")),
                      ("tokens_per_expert", torch.zeros(E - 1, dtype=torch.int32, device="cuda"))):
        args = dict(small, **{name: bad})
        with pytest.raises(ValueError):
            ep.ep_dispatch_layout_noalloc(ids10, 10, 10, K, E, R, **args)
    with pytest.raises(ValueError):
        ep.ep_dispatch_layout_noalloc(ids10, 10, 9, K, E, R, **small)      # N < T
    with pytest.raises(ValueError):
        ep.ep_dispatch_layout_noalloc(ids10[:5], 10, 10, K, E, R, **small)  # short ids
    torch.cuda.synchronize()
