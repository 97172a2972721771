"""Full-size workloads, in the launch configuration the benchmark times
(default permute, all SMs), plus the other permute implementation.

Every output is compared with the oracle, element by element:
- the layout (counts, prefix sums, every position) in full;
- every routed pair's receive row, score and source, against the oracle's
  definition recv_x[pos[t,k]] = x[t] (with pos already equal to the oracle's);
- the combine of EVERY token, in bf16 (bit for bit) and, from the same
  receive buffer, in fp32 before the cast (within 1e-6 relative and bit for
  bit), against the oracle's combine of the identity expert's rows, run on
  host threads in token slices.
"""
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_combine_equal, assert_layout_equal, oracle_combine_all, to_dev, to_np

pytestmark = pytest.mark.gpu


_WANT: dict = {}     # oracle outputs per (workload, source rank, dtype), shared by both impls


def oracle_out(orc, key, inp, pos, kind):
    if (key, kind) not in _WANT:
        _WANT[(key, kind)] = oracle_combine_all(orc, inp["x"], inp["scores"], pos, kind)
    return _WANT[(key, kind)]


def check_call(orc, buf, w, inp, N, key, fp32=True):
    x, ids, sc = inp["x"], inp["ids"], inp["scores"]
    T = ids.shape[0]
    xd, idd, scd = to_dev(x), to_dev(ids), to_dev(sc)
    d = buf.dispatch(xd, scd, idd, N)
    out = buf.combine(d.recv_x, scd)
    out32 = buf.combine(d.recv_x, scd, out_dtype=torch.float32) if fp32 else None
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
    del rows, tok, a, b, q
    # combine of every token, bf16 and fp32
    assert_combine_equal(to_np(out), oracle_out(orc, key, inp, ref["pos"], "same"))
    if fp32:
        assert_combine_equal(to_np(out32), oracle_out(orc, key, inp, ref["pos"], "f32"))
    del d, out, out32


@pytest.mark.parametrize("impl", [ep.EP_PERMUTE_DEFAULT, ep.EP_PERMUTE_VEC],
                         ids=["default", "vec"])
@pytest.mark.parametrize("name", ["mixtral", "deepseek", "prefill32k"])
def test_fullsize(orc, name, impl):
    w = W.WORKLOADS[name]
    inp = W.make(name)
    buf = ep.Buffer(w.N_max, w.D, w.E, w.R, w.K, dtype=torch.bfloat16, permute_impl=impl)
    check_call(orc, buf, w, inp, w.N, (name, 0))
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
        check_call(orc, buf, w, inp, N, ("ragged", r))
    assert buf.info()["workspace_bytes"] == ep.ep_buffer_required_bytes(buf.cfg)
    buf.close()
