"""Extreme and non-finite values through dispatch and combine, on every dispatch path.

- x drawn as uniformly random bit patterns: NaNs, infinities, subnormals,
  signed zeros and values near the overflow threshold all occur. The dispatch
  copies bytes, so every receive row equals the oracle's bit for bit, NaN
  payloads included.
- The combine and the backward equal the oracle bit for bit on every output,
  NaNs included: a NaN that the arithmetic produces is the canonical quiet NaN
  (7fc00000 in fp32, 7fc0 in bf16) on both sides, whatever NaN the inputs or
  the hardware carry (IEEE 754-2008 6.2 fixes only that the result is a quiet
  NaN; the one encoding is the reading taken).
- Rows made by hand for the bf16 overflow tie, a sum just below it, -0 + -0,
  inf - inf, a subnormal product (a flush to zero would show), 0 * inf and
  NaN operands with a sign, a payload or the signalling bit are checked
  against the values IEEE-754 arithmetic fixes, and against the oracle.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_expert_gb300 as ep
import workloads as W
from gpu_util import assert_layout_equal, assert_recv_equal, bits, to_dev, to_np, torch_dtype
from oracle_pins import bf16_is_nan, special_value_case, special_value_f32, special_value_y

pytestmark = pytest.mark.gpu

TAG_BITS = 31


def is_nan(a: np.ndarray) -> np.ndarray:
    return bf16_is_nan(a) if a.dtype == np.uint16 else np.isnan(a)


def assert_bits_equal(got: np.ndarray, want: np.ndarray) -> None:
    """Bit for bit, NaNs included; on a mismatch, says how many differ and
    whether NaNs are among them."""
    assert got.shape == want.shape and got.dtype == want.dtype
    bad = bits(got) != bits(want)
    if np.any(bad):
        n_nan = int((bad & is_nan(want)).sum())
        raise AssertionError(f"{int(bad.sum())} outputs differ from the oracle "
                             f"({n_nan} where the oracle's is a NaN)")


def random_bits(seed: int, T: int, D: int, dtype: str) -> np.ndarray:
    v = W.u64(seed, TAG_BITS, T * D).reshape(T, D)
    if dtype == "bf16":
        return (v & np.uint64(0xFFFF)).astype(np.uint16)
    return (v & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


CASES = {
    # name: (seed, T, N, D, dtype, E, K, R)
    "bf16": (160, 300, 302, 128, "bf16", 16, 4, 4),
    "f32": (161, 200, 200, 64, "f32", 8, 3, 2),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_random_bit_patterns(orc, path, case):
    seed, T, N, D, dtype, E, K, R = CASES[case]
    x = random_bits(seed, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, "zipf", "sigmoid_norm")
    sc[::7, 0] = 0.0          # 0 * inf and 0 * NaN occur too
    buf = ep.Buffer(N, D, E, R, K, dtype=torch_dtype(dtype), permute_impl=path)
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    outs = {"same": buf.combine(d.recv_x, scd)}
    if dtype == "bf16":
        outs["f32"] = buf.combine(d.recv_x, scd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    assert_layout_equal(d.layout, ref)
    assert_recv_equal(d, ref, R)
    n_nan = 0
    for kind, out in outs.items():
        want, err = orc.combine(ref["recv_x"], sc, ref["pos"], ref["rank_prefix"], ref["S"], R,
                                kind)
        assert err == 0
        assert_bits_equal(to_np(out), want)
        n_nan += int(is_nan(want).sum())
    assert n_nan > 0, "the inputs produced no NaN: the case tests nothing it claims"
    buf.close()


@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_ieee_special_values(orc, path, out_dtype):
    ids, sc, rows, want = special_value_case()
    T, D, E, R, K = ids.shape[0], 8, 2, 1, 2
    x = np.zeros((T, D), np.uint16)
    buf = ep.Buffer(T, D, E, R, K, dtype=torch.bfloat16, permute_impl=path)
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), T)
    ref = orc.dispatch(x, sc, ids, T, E, R)
    assert_layout_equal(d.layout, ref)
    y = special_value_y(ref, rows, D)
    od = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    out = to_np(buf.combine(to_dev(y), scd, out_dtype=od))
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    oracle_out, err = orc.combine(y, sc, ref["pos"], ref["rank_prefix"], ref["S"], R, out_dtype)
    assert err == 0
    assert_bits_equal(out, oracle_out)
    if out_dtype == "bf16":
        for t, w in enumerate(want):
            assert np.all(out[t] == w), (t, hex(int(out[t, 0])), hex(w))
    else:
        assert np.array_equal(out.view(np.uint32), special_value_f32(want, D))
    buf.close()


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_random_bit_patterns(orc, case):
    # grad_y = s * grad_out (one product, one rounding) and grad_x (the fma chain
    # with unit weights) against the oracle, bit for bit. The score gradients
    # (length-D dot products in a free fp32 order) are left out here: with
    # magnitudes up to the format's maximum, a partial fp32 sum can overflow where
    # the oracle's exact sum does not.
    seed, T, N, D, dtype, E, K, R = CASES[case]
    x = random_bits(seed, T, D, dtype)
    g = random_bits(seed + 1, T, D, dtype)
    ids, sc = W.routing(seed, T, E, K, "uniform", "sigmoid_norm")
    sc[::5, -1] = 0.0
    buf = ep.Buffer(N, D, E, R, K, dtype=torch_dtype(dtype))
    scd = to_dev(sc)
    d = buf.dispatch(to_dev(x), scd, to_dev(ids), N)
    grad_y, _ = buf.combine_backward(to_dev(g), d.recv_x, scd, want_scores=False)
    grad_x, _ = buf.dispatch_backward(grad_y, T)
    grad_x32, _ = buf.dispatch_backward(grad_y, T, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch(x, sc, ids, N, E, R)
    S = ref["S"]
    gy_ref, _, err = orc.combine_backward(g, ref["recv_x"], sc, ref["pos"], ref["rank_prefix"],
                                          S, R)
    assert err == 0
    pos = ref["pos"]
    valid = pos[pos >= 0]
    assert_bits_equal(to_np(grad_y.reshape(R * S, D))[valid], gy_ref[valid])
    for out, kind in ((grad_x, "same"), (grad_x32, "f32")):
        want, _, _ = orc.dispatch_backward(gy_ref, None, pos, ref["rank_prefix"], S, R, kind)
        assert_bits_equal(to_np(out), want)
    buf.close()


def test_dedup_random_bit_patterns(orc):
    # The dedupe rows and their expansion are copies: bit for bit, NaN payloads
    # included; the combine on the expanded rows as above.
    seed, T, N, D, dtype, E, K, R = CASES["bf16"]
    x = random_bits(seed + 7, T, D, dtype)
    ids, sc = W.routing(seed + 7, T, E, K, "zipf", "sigmoid_norm")
    buf = ep.Buffer(N, D, E, R, K, dtype=torch.bfloat16)
    scd, idd = to_dev(sc), to_dev(ids)
    dd = buf.dispatch_dedup(to_dev(x), scd, idd, N)
    y = buf.dedup_expand(idd)
    out = buf.combine(y, scd)
    torch.cuda.synchronize()
    assert buf.device_error() == 0
    ref = orc.dispatch_dedup(x, sc, ids, N, E, R)
    P, tir = ref["P"], ref["tokens_in_rank"]
    rx = to_np(dd.recv_x.reshape(R * P, D))
    for r in range(R):
        rows = slice(r * P, r * P + int(tir[r]))
        assert np.array_equal(bits(rx[rows]), bits(ref["recv_tok_x"][rows]))
    d = orc.dispatch(x, sc, ids, N, E, R)
    valid = d["pos"][d["pos"] >= 0]
    assert np.array_equal(bits(to_np(y.reshape(-1, D))[valid]), bits(d["recv_x"][valid]))
    want, _ = orc.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
    assert_bits_equal(to_np(out), want)
    buf.close()
