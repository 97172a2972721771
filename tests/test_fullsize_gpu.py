"""Full-size workloads, in the launch configuration the benchmark times
(default permute, all SMs), plus the other permute implementation.

The layout (counts, prefix sums, every position) is compared with the oracle
in full. Receive rows are checked for every routed pair against the oracle's
definition recv_x[pos[t,k]] = x[t] (with pos already equal to the oracle's).
Combine is checked bit for bit on a sample of tokens the oracle computes one
by one (first, last and seeded-random tokens).
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_combine_equal, assert_layout_equal, sampled_combine_ref, to_dev, to_np

pytestmark = pytest.mark.gpu


def check_call(orc, buf, w, inp, N, n_sample=160):
    x, ids, sc = inp["x"], inp["ids"], inp["scores"]
    T = ids.shape[0]
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, N)
    out = buf.combine(d.recv_x, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.layout(ids, N, w.E, w.R)
    assert_layout_equal(d.layout, ref)
    # every routed pair's row, score and source, compared on the device
    pos = d.layout.pos.reshape(-1).long()
    valid = pos >= 0
    rows = d.recv_x.reshape(-1, w.D)[pos[valid]]
    tok = torch.arange(T, device="cuda").repeat_interleave(w.K)[valid]
    a = rows.view(torch.int16) if rows.dtype == torch.bfloat16 else rows.view(torch.int32)
    b = xd[tok].view(torch.int16) if xd.dtype == torch.bfloat16 else xd[tok].view(torch.int32)
    assert torch.equal(a, b), "receive rows differ from x"
    assert torch.equal(d.recv_scores.reshape(-1)[pos[valid]], scd.reshape(-1)[valid])
    q = torch.arange(T * w.K, device="cuda", dtype=torch.int32)[valid]
    assert torch.equal(d.recv_src.reshape(-1)[pos[valid]], q)
    # combine on a sample of tokens
    rng = np.random.default_rng(T)
    sample = np.unique(np.concatenate([np.arange(min(T, 48)), np.arange(max(0, T - 48), T),
                                       rng.integers(0, T, n_sample - 96)]))
    y = to_np(d.recv_x.reshape(-1, w.D))
    want = sampled_combine_ref(orc, y, sc, ref["pos"], sample)
    assert_combine_equal(to_np(out)[sample], want)
    del d, out, rows


@pytest.mark.parametrize("impl", [ep.EP_PERMUTE_DEFAULT, ep.EP_PERMUTE_VEC],
                         ids=["default", "vec"])
@pytest.mark.parametrize("name", ["mixtral", "deepseek", "prefill32k"])
def test_fullsize(orc, name, impl):
    w = W.WORKLOADS[name]
    inp = W.make(name)
    buf = ep.Buffer(w.N_max, w.D, w.E, w.R, w.K, dtype=torch.bfloat16, permute_impl=impl)
    check_call(orc, buf, w, inp, w.N)
    buf.close()
    del buf
    torch.cuda.empty_cache()


def test_ragged_eight_source_ranks(orc):
    # Eight logical source ranks with unaligned counts in [41, 3543], each
    # dispatched with the EP-group max padded to 4, through one buffer sized
    # from num_max_tokens_per_rank = 4096.
    w = W.WORKLOADS["ragged"]
    counts = W.ragged_counts(w)
    N = max(counts)
    buf = ep.Buffer(w.N_max, w.D, w.E, w.R, w.K, dtype=torch.bfloat16)
    for r in range(w.ragged_ranks):
        inp = W.make("ragged", rank=r)
        assert inp["T"] == counts[r] and counts[r] % 4 != 0
        check_call(orc, buf, w, inp, N, n_sample=120)
    assert buf.info()["workspace_bytes"] == ep.ep_buffer_required_bytes(buf.cfg)
    buf.close()
