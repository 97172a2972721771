"""The seeded input generator: determinism, shapes and the stated distributions."""
import numpy as np

import workloads as W


def test_splitmix64_known_values():
    # splitmix64 from state 0: the first outputs are the published sequence
    # 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F.
    base = np.uint64(0)
    G = np.uint64(0x9E3779B97F4A7C15)
    with np.errstate(over="ignore"):
        z = np.array([base + G, base + G * np.uint64(2), base + G * np.uint64(3)], np.uint64)
        got = [int(v) for v in W._mix64(z)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_stream_independent():
    a = W.make("tiny")
    b = W.make("tiny")
    assert np.array_equal(a["x"], b["x"]) and np.array_equal(a["ids"], b["ids"])
    assert np.array_equal(a["scores"], b["scores"])
    c = W.make("tiny", seed=123)
    assert not np.array_equal(a["x"], c["x"])
    # chunked generation equals one pass
    assert np.array_equal(W.uniform(3, 1, 10, start=5), W.uniform(3, 1, 15)[5:])


def test_shapes_and_ranges():
    for name in ("tiny", "mixtral"):
        d = W.make(name)
        w = d["workload"]
        assert d["x"].shape == (w.T, w.D)
        assert d["x"].dtype == (np.uint16 if w.dtype == "bf16" else np.float32)
        assert d["ids"].shape == (w.T, w.K) and d["ids"].dtype == np.int32
        assert d["ids"].min() >= 0 and d["ids"].max() < w.E
        for row in d["ids"]:
            assert len(set(row.tolist())) == w.K           # drawn without replacement


def test_score_kinds():
    ids = W.topk_ids_uniform(1, 500, 8, 2)
    s = W.topk_scores(1, ids, 8, "softmax_topk")
    assert np.allclose(s.sum(1), 1.0, atol=1e-6)
    s = W.topk_scores(1, ids, 8, "softmax_all")
    assert np.all(s.sum(1) < 1.0) and np.all(s > 0)            # not renormalised
    ids = W.topk_ids_uniform(1, 500, 256, 8)
    s = W.topk_scores(1, ids, 256, "sigmoid_norm")
    assert np.allclose(s.sum(1), 1.0, atol=1e-6)


def test_zipf_skew():
    ids = W.topk_ids_zipf(2, 4000, 256, 8)
    cnt = np.bincount(ids.ravel(), minlength=256)
    assert cnt[0] > cnt[10] > cnt[200]
    # The first draw of a weighted draw without replacement picks expert e with
    # probability w_e / sum(w): check it for the hottest expert (4 sigma).
    w = (np.arange(256) + 1.0) ** -1.1
    p0 = w[0] / w.sum()
    frac = float(np.mean(ids[:, 0] == 0))
    assert abs(frac - p0) < 4 * np.sqrt(p0 * (1 - p0) / 4000)
    assert cnt[0] > 0.75 * 4000                  # most tokens pick expert 0 somewhere
    for row in ids[:200]:
        assert len(set(row.tolist())) == 8


def test_ragged_counts():
    w = W.WORKLOADS["ragged"]
    c = W.ragged_counts(w)
    assert len(c) == 8
    assert all(41 <= v <= 3543 and v % 4 != 0 for v in c)


def test_normal_moments():
    v = W.normal(7, 1, 200_000)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
