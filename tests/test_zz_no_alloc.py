"""ep_dispatch_layout_noalloc: the dispatch layout for callers that cannot
allocate device memory (for example an op inside a host framework that owns
every device allocation and only hands it input and output tensors). It takes
the ids and caller-owned outputs and uses a fixed library-owned device array
for its tile tables, so it never allocates.

Its results must equal those of the buffer-based ep_dispatch_layout. This file
is named to be collected last, so a failure here leaves every other test run.
"""
import ctypes as C

import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
from combine_topk_ids_expert_gb300 import _abi
import workloads as W

FIELDS = ("tokens_per_expert", "expert_offset", "rows_per_rank", "rank_prefix",
          "tokens_in_rank", "pos")


def poisoned_outputs(T, K, E, R):
    def full(*shape):
        return torch.full(shape, -7, dtype=torch.int32, device="cuda")
    return {"tokens_per_expert": full(E), "expert_offset": full(E), "rows_per_rank": full(R),
            "rank_prefix": full(R), "tokens_in_rank": full(R), "pos": full(T, K)}


@pytest.mark.gpu
def test_noalloc_layout_matches_buffer_layout_on_two_calls():
    E, K, R = 256, 8, 8
    # Two calls in a row through the C ABI: a ragged multi-tile call with
    # padding, then the full DeepSeek-shaped routing (Zipf ids, 8192 tokens).
    calls = [(W.topk_ids_zipf(51, 1000, E, K), 1003),
             (W.topk_ids_zipf(W.WORKLOADS["deepseek"].seed, 8192, E, K), 8192)]
    buf = ep.Buffer(8192, 64, E, R, K, dtype=torch.bfloat16)
    for ids_np, N in calls:
        ids = torch.from_numpy(ids_np).cuda()
        T = ids.shape[0]
        lay = buf.dispatch_layout(ids, N)
        out = poisoned_outputs(T, K, E, R)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ep.ep_dispatch_layout_noalloc(ids, T, N, K, E, R, **out, error_flags=err)
        torch.cuda.synchronize()
        for name in FIELDS:   # integer results: bit-exact, as for every layout test
            assert torch.equal(out[name], getattr(lay, name)), name
        assert int(err.item()) == 0
        assert buf.device_error() == 0
    buf.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # Rejected on the host before any device work: 600k tokens at E=256, K=8
    # need 2344 tiles of tables, more than the 4 MiB array holds (2016).
    L = _abi.lib()
    st = L.ep_dispatch_layout_noalloc(None, 600_000, 600_000, 8, 256, 8, None, None, None, None,
                                      None, None, None, None)
    assert st == _abi.EP_ERR_INVALID_ARG          # null outputs are refused first
    fake = C.c_void_p(0x1000)
    st = L.ep_dispatch_layout_noalloc(fake, 600_000, 600_000, 8, 256, 8, fake, fake, fake, fake,
                                      fake, fake, None, None)
    assert st == _abi.EP_ERR_CAPACITY
    st = L.ep_dispatch_layout_noalloc(fake, 130_000, 130_000, 8, 1024, 64, fake, fake, fake,
                                      fake, fake, fake, None, None)
    assert st == _abi.EP_ERR_CAPACITY
