"""ep_pattern_probe, the measurement aid behind `bench.py --mode ceilings`:
each access pattern moves exactly the rows it names (checked against numpy on
small cases with ragged row counts), so the ceilings it times are of real
copies, fan-outs and gathers."""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep

pytestmark = pytest.mark.gpu


def _xor_rows(a: np.ndarray) -> np.ndarray:
    """XOR of each row's 16-byte words: [rows, 4] int32."""
    return np.bitwise_xor.reduce(a.reshape(a.shape[0], -1, 4), axis=1)


@pytest.mark.parametrize("rows,row_bytes,fan", [(37, 2 * 7168, 8), (5, 16, 3), (300, 8192, 2)])
def test_patterns_move_the_rows_they_name(rows, row_bytes, fan):
    rng = np.random.default_rng(rows)
    n = row_bytes // 4
    src_np = rng.integers(-2**31, 2**31 - 1, size=(fan * rows, n), dtype=np.int64).astype(np.int32)
    src = torch.from_numpy(src_np).cuda()
    dst = torch.zeros((fan * rows, n), dtype=torch.int32, device="cuda")
    ep.ep_pattern_probe(ep._abi.EP_PATTERN_COPY, src, dst, rows, row_bytes)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy()[:rows], src_np[:rows])
    assert not dst[rows:].any()
    dst.zero_()
    ep.ep_pattern_probe(ep._abi.EP_PATTERN_FANOUT, src, dst, rows, row_bytes, fan)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().reshape(fan, rows, n)
    for j in range(fan):
        assert np.array_equal(got[j], src_np[:rows]), j
    dst.zero_()
    ep.ep_pattern_probe(ep._abi.EP_PATTERN_GATHER, src, dst, rows, row_bytes, fan)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(src_np.reshape(fan, rows, n), axis=0)
    assert np.array_equal(dst.cpu().numpy()[:rows], want)
    dst.zero_()
    ep.ep_pattern_probe(ep._abi.EP_PATTERN_READ, src, dst, rows, row_bytes)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().reshape(-1)[:rows * 4].reshape(rows, 4)
    assert np.array_equal(got, _xor_rows(src_np[:rows]))
    dst.zero_()
    ep.ep_pattern_probe(ep._abi.EP_PATTERN_WRITE, None, dst, rows, row_bytes)
    torch.cuda.synchronize()
    got = dst.cpu().numpy()[:rows].reshape(rows, -1, 4)
    r = np.arange(rows)[:, None]
    v = np.arange(row_bytes // 16)[None, :]
    assert np.array_equal(got[:, :, 0], np.broadcast_to(r, got.shape[:2]))
    assert np.array_equal(got[:, :, 1], np.broadcast_to(v, got.shape[:2]))
    assert not dst[rows:].any()


def test_pattern_probe_rejects_bad_arguments():
    t = torch.zeros(64, dtype=torch.int32, device="cuda")
    L = ep._abi.lib()
    bad = [(ep._abi.EP_PATTERN_COPY, 4, 24, 1),      # row bytes not a multiple of 16
           (7, 4, 16, 1),                           # no such pattern
           (ep._abi.EP_PATTERN_FANOUT, 1, 16, 0),   # fan < 1
           (ep._abi.EP_PATTERN_GATHER, 1, 16, 65)]  # fan > 64
    for pat, rows, rb, fan in bad:
        assert L.ep_pattern_probe(pat, t.data_ptr(), t.data_ptr(), rows, rb, fan, None) == \
            ep._abi.EP_ERR_INVALID_ARG
    assert L.ep_pattern_probe(ep._abi.EP_PATTERN_COPY, t.data_ptr() + 4, t.data_ptr(), 1, 16, 1,
                              None) == ep._abi.EP_ERR_ALIGNMENT
    with pytest.raises(ValueError):
        ep.ep_pattern_probe(ep._abi.EP_PATTERN_FANOUT, t, t, 4, 64, 2)   # dst too small
