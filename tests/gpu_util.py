"""Helpers shared by the GPU parity tests: numpy <-> torch and oracle comparisons."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

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


# Host threads for full-size oracle runs: each thread runs the single-threaded
# oracle on its own slice of tokens (ctypes releases the GIL during the call).
ORACLE_THREADS = max(1, min(16, os.cpu_count() or 1))


def pool_map(fn, items):
    with ThreadPoolExecutor(ORACLE_THREADS) as ex:
        return list(ex.map(fn, items))


def identity_block(x: np.ndarray, pos: np.ndarray, a: int, b: int):
    """Tokens [a, b) of a call under the identity expert, as a problem of its own:
    the receive rows their valid pairs land on (y[pos[t, k]] = x[t]) packed in
    flat pair order into one rank. Returns (rows, cpos, rank_prefix, S) for the
    oracle; cpos[t - a, k] is the pair's row in the block or -1. Each token's
    combine and backward depend only on its own pairs' rows, so the oracle run
    on the block gives exactly its run on the whole call for these tokens."""
    p = pos[a:b]
    valid = p >= 0
    n = int(valid.sum())
    cpos = np.full(p.shape, -1, np.int32)
    cpos[valid] = np.arange(n, dtype=np.int32)
    tok = np.repeat(np.arange(a, b), p.shape[1]).reshape(p.shape)[valid]
    rows = x[tok] if n else np.zeros((1, x.shape[1]), x.dtype)
    return rows, cpos, np.array([n], np.int32), max(n, 1)


def oracle_combine_all(o: oracle.Oracle, x: np.ndarray, scores: np.ndarray, pos: np.ndarray,
                       out_dtype: str = "same", chunk: int = 1024) -> np.ndarray:
    """The oracle's combine of EVERY token of a call whose expert is the identity
    (pos: the oracle's own positions), run in token slices on host threads."""
    T = pos.shape[0]

    def run(a):
        rows, cpos, prefix, S = identity_block(x, pos, a, min(T, a + chunk))
        out, err = o.combine(rows, scores[a:a + chunk], cpos, prefix, S, 1, out_dtype)
        assert err == 0
        return out

    parts = pool_map(run, range(0, T, chunk))
    if parts:
        return np.concatenate(parts)
    kind = x.dtype if out_dtype == "same" else (np.uint16 if out_dtype == "bf16" else np.float32)
    return np.zeros((0, x.shape[1]), kind)


def oracle_backward_all(o: oracle.Oracle, x: np.ndarray, g: np.ndarray, scores: np.ndarray,
                        pos: np.ndarray, chunk: int = 1024):
    """The oracle's backward of EVERY token of an identity-expert call: grad_y of
    the valid pairs in flat pair order [n_valid, D], grad_scores [T, K], grad_x
    [T, D] (dispatch backward of the oracle's own grad_y)."""
    T = pos.shape[0]

    def run(a):
        b = min(T, a + chunk)
        rows, cpos, prefix, S = identity_block(x, pos, a, b)
        gy, gs, err = o.combine_backward(g[a:b], rows, scores[a:b], cpos, prefix, S, 1)
        assert err == 0
        gx, _, err = o.dispatch_backward(gy, None, cpos, prefix, S, 1)
        assert err == 0
        return gy[:int(prefix[0])], gs, gx

    parts = pool_map(run, range(0, T, chunk))
    return (np.concatenate([q[0] for q in parts]), np.concatenate([q[1] for q in parts]),
            np.concatenate([q[2] for q in parts]))


def valid_rows(t: torch.Tensor, pos: np.ndarray) -> np.ndarray:
    """Rows of a receive-layout tensor at every valid position, in flat pair
    order, gathered on the device and copied to the host."""
    D = t.shape[-1]
    p = torch.from_numpy(pos.reshape(-1)[pos.reshape(-1) >= 0].astype(np.int64)).cuda()
    return to_np(t.reshape(-1, D)[p])
