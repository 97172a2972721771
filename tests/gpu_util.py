"""Helpers shared by the GPU parity tests: numpy <-> torch and oracle comparisons."""
from __future__ import annotations

import numpy as np
import torch

import combine_topk_ids_expert_gb300 as ep
import oracle
import workloads as W


def to_dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_np(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy; bf16 comes back as uint16 bit patterns."""
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def torch_dtype(kind: str) -> torch.dtype:
    return torch.bfloat16 if kind == "bf16" else torch.float32


LAYOUT_FIELDS = [("cnt", "tokens_per_expert"), ("expert_offset", "expert_offset"),
                 ("rows_per_rank", "rows_per_rank"), ("rank_prefix", "rank_prefix"),
                 ("tokens_in_rank", "tokens_in_rank"), ("pos", "pos")]


def assert_layout_equal(lay: ep.Layout, ref: dict) -> None:
    for rname, gname in LAYOUT_FIELDS:
        got = to_np(getattr(lay, gname))
        assert np.array_equal(got, ref[rname]), f"{gname} differs from the oracle"
    assert lay.rank_stride == ref["S"]


def assert_recv_equal(d: ep.DispatchResult, ref: dict, R: int) -> None:
    """Every defined receive row (inside each rank's true total; for the packed
    layout, every row below the true total) equals the oracle's, bit for bit (NaN
    payloads and signed zeros included: the rows are copies)."""
    S = ref["S"]
    rx = to_np(d.recv_x.reshape(R * S, -1))
    rs = to_np(d.recv_scores.reshape(-1))
    rsrc = to_np(d.recv_src.reshape(-1))
    if d.layout.packed:     # ranks back to back: rows [0, true total)
        ranges = [(0, int(ref["rank_prefix"][-1]))]
    else:                   # rank r: rows [r*S, r*S + rows_per_rank[r])
        ranges = [(r * S, r * S + int(ref["rows_per_rank"][r])) for r in range(R)]
    for r, (lo, hi) in enumerate(ranges):
        assert np.array_equal(bits(rx[lo:hi]), bits(ref["recv_x"][lo:hi])), f"recv_x rank {r}"
        assert np.array_equal(rs[lo:hi].view(np.uint32),
                              ref["recv_scores"][lo:hi].view(np.uint32)), f"recv_scores rank {r}"
        assert np.array_equal(rsrc[lo:hi], ref["recv_src"][lo:hi]), f"recv_src rank {r}"


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


def assert_combine_equal(got: np.ndarray, want: np.ndarray) -> None:
    """bf16 and fp32 combine outputs must match bit for bit (same fma chain);
    the fp32 check also states the 1e-6 relative bound explicitly."""
    assert got.shape == want.shape and got.dtype == want.dtype
    if got.dtype == np.float32:
        diff = np.abs(got.astype(np.float64) - want.astype(np.float64))
        scale = np.maximum(np.abs(want.astype(np.float64)), 1e-30)
        assert np.all(diff <= 1e-6 * scale), f"max rel diff {np.max(diff / scale)}"
    assert np.array_equal(bits(got), bits(want)), "combine differs from the oracle bitwise"


def sampled_combine_ref(o: oracle.Oracle, y: np.ndarray, scores: np.ndarray, pos: np.ndarray,
                        tokens: np.ndarray, out_dtype: str = "same") -> np.ndarray:
    """Oracle combine for a sample of tokens: their gathered rows are packed into a
    compact one-rank receive block and the oracle runs its definition on it."""
    K = pos.shape[1]
    n = len(tokens)
    rows = []
    cpos = np.full((n, K), -1, np.int32)
    for i, t in enumerate(tokens):
        for k in range(K):
            p = pos[t, k]
            if p >= 0:
                cpos[i, k] = len(rows)
                rows.append(y[p])
    ybuf = np.stack(rows) if rows else np.zeros((1, y.shape[1]), y.dtype)
    S = max(1, len(rows))
    out, err = o.combine(ybuf, scores[tokens], cpos, np.array([len(rows)], np.int32), S, 1,
                         out_dtype)
    assert err == 0
    return out


def make_inputs(name: str, T: int | None = None, seed: int | None = None, rank: int = 0,
                replay: int | None = None, D: int | None = None):
    """Workload inputs; D overrides the hidden size for oracle-sized parity cases."""
    inp = W.make(name, T=T, seed=seed, rank=rank, replay=replay, with_x=(D is None))
    w = inp["workload"]
    if D is not None:
        base = w.seed if seed is None else seed
        inp["x"] = W.hidden(base + 7919 * rank, inp["T"], D, w.dtype)
    return inp
