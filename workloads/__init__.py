"""Seeded synthetic inputs for MoE token dispatch and combine.

This module makes what a router hands to a token dispatcher, and nothing else:
hidden rows ``x_TD``, top-k expert ids ``topk_expert_ids_TK`` and top-k scores
``topk_scores_TK``, with the shapes and value distributions of the workloads
the dispatcher pages describe. It holds none of the dispatch/combine
arithmetic (no padding, counting, placement, weighting or result rounding), so
the CUDA path's tests, the CPU oracle's tests and the benchmark can all draw
from it without sharing any part of the method.

Random numbers come from splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator: output i of a stream with base ``b`` is ``mix64(b + (i + 1) * G)``
with ``G = 0x9E3779B97F4A7C15``. Uniforms take the top 53 bits; normals use the
Box-Muller transform; bf16 values are fp32 normals truncated to their top 16
bits (a distribution choice, not a rounding the method performs).

The integer streams are bit-reproducible everywhere. The float transforms go
through numpy's log/cos/sin, whose last ulp may differ between CPU families, so
tests always feed the SAME generated arrays to both sides within one process
and never store generated values as expected results.

Workloads (sizes from the pages' settings; see ``WORKLOADS``):
  tiny        T=16, D=64 fp32, E=8, K=2, R=2, N=16 (N_max=32); uniform ids,
              scores = softmax over all 8 N(0,1) logits gathered at the ids.
  mixtral     T=4096, D=4096 bf16, E=8, K=2, R=1, N=N_max=4096; uniform ids,
              scores = softmax over the 2 chosen N(0,1) logits.
  deepseek    T=8192, D=7168 bf16, E=256, K=8, R=8, N=N_max=8192; ids drawn
              without replacement with weight (e+1)^-1.1 (Zipf s=1.1),
              scores = sigmoid(z_k) / sum_j sigmoid(z_j), z ~ N(0,1).
  ragged      8 logical source ranks with T_r ~ U[41, 3543], T_r % 4 != 0,
              D=7168 bf16, E=256, K=8, R=8, N_max=4096; uniform ids,
              sigmoid-normalised scores.
  prefill32k  T=32768, D=7168 bf16, E=256, K=8, R=8, N=N_max=32768; fixed x,
              fresh Zipf(1.1) ids and sigmoid scores for every replay.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TAG_MUL = np.uint64(0xD1B54A32D192ED03)

# Stream tags: one independent stream per purpose.
TAG_X, TAG_IDS, TAG_LOGITS, TAG_COUNTS = 1, 2, 3, 4

_CHUNK = 1 << 23  # values generated per numpy pass (bounds temporaries)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        v = np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (np.uint64(tag) * _TAG_MUL)],
                     dtype=np.uint64)
        return _mix64(v)[0]


def u64(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start..start+n-1 of the splitmix64 stream (seed, tag)."""
    base = _stream_base(seed, tag)
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix64(base + ctr * _GAMMA)


def uniform(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    """Uniform float64 in [0, 1) from the top 53 bits."""
    return (u64(seed, tag, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    """N(0, 1) float64 by Box-Muller; pair i of uniforms gives outputs 2i, 2i+1."""
    out = np.empty(n, dtype=np.float64)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        m = min(_CHUNK, npairs - p0)
        u = uniform(seed, tag, 2 * m, start=2 * p0)
        u1 = 1.0 - u[0::2]          # in (0, 1]
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = 2.0 * np.pi * u2
        blk = np.empty(2 * m, dtype=np.float64)
        blk[0::2] = r * np.cos(th)
        blk[1::2] = r * np.sin(th)
        lo = 2 * p0
        hi = min(n, lo + 2 * m)
        out[lo:hi] = blk[: hi - lo]
    return out


def bf16_bits_trunc(a32: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) holding the top 16 bits of fp32 values."""
    return (np.ascontiguousarray(a32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@dataclass(frozen=True)
class Workload:
    name: str
    D: int
    dtype: str          # "bf16" or "f32"
    E: int
    K: int
    R: int
    N_max: int
    T: int | None       # None: per-rank counts drawn (ragged)
    N: int | None       # num_tokens_per_rank when fixed by the setting
    ids: str            # "uniform" or "zipf"
    scores: str         # "softmax_all", "softmax_topk" or "sigmoid_norm"
    seed: int
    graph_replays: int = 0
    ragged_ranks: int = 0
    ragged_lo: int = 0
    ragged_hi: int = 0

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


_SEED0 = 0xE9D15000

WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", D=64, dtype="f32", E=8, K=2, R=2, N_max=32, T=16, N=16,
                     ids="uniform", scores="softmax_all", seed=_SEED0 + 0),
    "mixtral": Workload("mixtral", D=4096, dtype="bf16", E=8, K=2, R=1, N_max=4096, T=4096,
                        N=4096, ids="uniform", scores="softmax_topk", seed=_SEED0 + 1),
    "deepseek": Workload("deepseek", D=7168, dtype="bf16", E=256, K=8, R=8, N_max=8192,
                         T=8192, N=8192, ids="zipf", scores="sigmoid_norm", seed=_SEED0 + 2),
    "ragged": Workload("ragged", D=7168, dtype="bf16", E=256, K=8, R=8, N_max=4096, T=None,
                       N=None, ids="uniform", scores="sigmoid_norm", seed=_SEED0 + 3,
                       ragged_ranks=8, ragged_lo=41, ragged_hi=3543),
    "prefill32k": Workload("prefill32k", D=7168, dtype="bf16", E=256, K=8, R=8, N_max=32768,
                           T=32768, N=32768, ids="zipf", scores="sigmoid_norm",
                           seed=_SEED0 + 4, graph_replays=100),
}

ZIPF_S = 1.1


def hidden(seed: int, T: int, D: int, dtype: str) -> np.ndarray:
    """x_TD: N(0,1) rows; float32 [T, D] or bf16 bit patterns uint16 [T, D]."""
    v = normal(seed, TAG_X, T * D).astype(np.float32).reshape(T, D)
    return bf16_bits_trunc(v) if dtype == "bf16" else v


def topk_ids_uniform(seed: int, T: int, E: int, K: int) -> np.ndarray:
    """K distinct experts per token, uniform without replacement (int32 [T, K])."""
    keys = uniform(seed, TAG_IDS, T * E).reshape(T, E)
    order = np.argsort(keys, axis=1, kind="stable")[:, :K]
    return np.ascontiguousarray(order, dtype=np.int32)


def topk_ids_zipf(seed: int, T: int, E: int, K: int, s: float = ZIPF_S) -> np.ndarray:
    """K distinct experts per token by weighted draws without replacement,
    weight of expert e proportional to (e + 1)^-s. Efraimidis-Spirakis keys
    log(u) / w: the K largest, in decreasing key order, have the distribution of
    K sequential weighted draws. Expert 0 is the hottest."""
    w = (np.arange(E, dtype=np.float64) + 1.0) ** (-s)
    u = 1.0 - uniform(seed, TAG_IDS, T * E).reshape(T, E)   # (0, 1]
    keys = np.log(u) / w[None, :]
    order = np.argsort(-keys, axis=1, kind="stable")[:, :K]
    return np.ascontiguousarray(order, dtype=np.int32)


def topk_scores(seed: int, ids: np.ndarray, E: int, kind: str) -> np.ndarray:
    """Router scores for the chosen ids (float32 [T, K])."""
    T, K = ids.shape
    if kind == "softmax_all":
        logits = normal(seed, TAG_LOGITS, T * E).reshape(T, E)
        ex = np.exp(logits - logits.max(axis=1, keepdims=True))
        p = ex / ex.sum(axis=1, keepdims=True)
        out = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    elif kind == "softmax_topk":
        z = normal(seed, TAG_LOGITS, T * K).reshape(T, K)
        ex = np.exp(z - z.max(axis=1, keepdims=True))
        out = ex / ex.sum(axis=1, keepdims=True)
    elif kind == "sigmoid_norm":
        z = normal(seed, TAG_LOGITS, T * K).reshape(T, K)
        sg = 1.0 / (1.0 + np.exp(-z))
        out = sg / sg.sum(axis=1, keepdims=True)
    else:
        raise ValueError(f"unknown score kind {kind!r}")
    return np.ascontiguousarray(out, dtype=np.float32)


def routing(seed: int, T: int, E: int, K: int, ids_kind: str, scores_kind: str):
    if ids_kind == "uniform":
        ids = topk_ids_uniform(seed, T, E, K)
    elif ids_kind == "zipf":
        ids = topk_ids_zipf(seed, T, E, K)
    else:
        raise ValueError(f"unknown id kind {ids_kind!r}")
    return ids, topk_scores(seed, ids, E, scores_kind)


def ragged_counts(w: Workload) -> list[int]:
    """Per-source-rank token counts T_r ~ U[lo, hi], redrawn while T_r % 4 == 0."""
    counts = []
    ctr = 0
    span = w.ragged_hi - w.ragged_lo + 1
    for _ in range(w.ragged_ranks):
        while True:
            v = w.ragged_lo + int(uniform(w.seed, TAG_COUNTS, 1, start=ctr)[0] * span)
            ctr += 1
            if v % 4 != 0:
                counts.append(v)
                break
    return counts


def make(name: str, *, T: int | None = None, seed: int | None = None, rank: int = 0,
         replay: int | None = None, with_x: bool = True) -> dict:
    """Inputs of one dispatch call of workload ``name``.

    ``T`` overrides the token count (smaller parity cases of the same shape);
    ``rank`` picks the source rank of the ragged workload; ``replay`` gives the
    fresh routing of a graph replay (x stays the workload's fixed x).
    Returns {"x", "ids", "scores", "T", "workload"}; x is None when with_x=False.
    """
    w = WORKLOADS[name]
    base = w.seed if seed is None else seed
    if T is None:
        T = ragged_counts(w)[rank] if w.T is None else w.T
    rseed = base + 7919 * rank
    x = hidden(rseed, T, w.D, w.dtype) if with_x else None
    if replay is not None:
        rseed = rseed + 1000 * (replay + 1)
    ids, scores = routing(rseed, T, w.E, w.K, w.ids, w.scores)
    return {"x": x, "ids": ids, "scores": scores, "T": T, "workload": w}
