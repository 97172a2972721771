"""Pins that tie the CPU oracle to facts outside itself.

Each pin takes an oracle build and raises AssertionError when the build
disagrees with: values the pages print (fixtures under tests/golden/, each
cited), closed forms, a library routine computing the same quantity another
way (numpy's stable sort and bincount, torch's bf16 cast), brute force on tiny
inputs, or an exact result within the fp32 error bound. test_oracle_pins.py
runs them against the real oracle; test_oracle_mutants.py runs them against
deliberately broken oracle builds and requires every break to be caught.
"""
from __future__ import annotations

import json
import os

import numpy as np

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _ids(seed, T, E, K):
    return W.topk_ids_uniform(seed, T, E, K)


def _exact_inputs(seed, T, D, K):
    """Hidden rows and scores whose fp32 products and K-term sums are exact:
    x = i/8 with |i| <= 64 (exact in bf16), scores = j/64 with 0 <= j <= 64."""
    xi = (W.u64(seed, 11, T * D) % np.uint64(129)).astype(np.int64) - 64
    x = (xi.astype(np.float32) / np.float32(8.0)).reshape(T, D)
    sj = (W.u64(seed, 12, T * K) % np.uint64(65)).astype(np.float32)
    return x, (sj / np.float32(64.0)).reshape(T, K)


def _bf16_bits(a32):
    """bf16 bit patterns of fp32 values that are exactly representable."""
    b = np.ascontiguousarray(a32, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def _f32_from_bits(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Padding and capacity: worked values from the pages
# ---------------------------------------------------------------------------

def pin_padding_vectors(o):
    g = _golden("padding_vectors.json")
    for c in g["single"]:
        assert o.pad_tokens(c["n"]) == c["padded"], c
    for c in g["group"]:
        assert o.pad_tokens(max(c["counts"])) == c["padded"], c


def pin_padding_closed_form(o):
    # Smallest multiple of 4 not below n, for every n in a range.
    for n in range(0, 200):
        p = o.pad_tokens(n)
        assert p % 4 == 0 and n <= p < n + 4, (n, p)


def pin_capacity(o):
    g = _golden("capacity.json")
    for c in g["pretrain"]:
        got = o.num_max_tokens_pretrain(c["local_batch_size"], c["seq_len"], c["cp"], c["tp"])
        assert got == c["expect"], (c, got)
    for c in g["inference"]:
        got = o.num_max_tokens_inference(c["max_num_batched_tokens"], c["cp"], c["tp"])
        assert got == c["expect"], (c, got)


def pin_rank_stride(o):
    # Worst case for one rank: every pair of every padded token lands there.
    for N, K in [(13, 2), (16, 2), (8192, 8), (3543, 8), (1, 1), (0, 4)]:
        assert o.rank_stride(N, K) == ((N + 3) // 4) * 4 * K, (N, K)


# ---------------------------------------------------------------------------
# bf16 rounding: hand-worked IEEE cases and torch's cast
# ---------------------------------------------------------------------------

def pin_bf16_golden(o):
    for f_hex, h_hex, why in _golden("bf16_rne.json")["cases"]:
        f = np.array([int(f_hex, 16)], dtype=np.uint32).view(np.float32)
        got = int(o.bf16_from_f32(f)[0])
        assert got == int(h_hex, 16), (f_hex, h_hex, hex(got), why)


def pin_bf16_nan_golden(o):
    # NaN conversions worked by hand from IEEE 754-2008 6.2.3 (sign and leading
    # payload bits kept, quiet bit set).
    for f_hex, h_hex, why in _golden("bf16_nan.json")["cases"]:
        f = np.array([int(f_hex, 16)], dtype=np.uint32).view(np.float32)
        got = int(o.bf16_from_f32(f)[0])
        assert got == int(h_hex, 16), (f_hex, h_hex, hex(got), why)


def pin_bf16_from_f64_golden(o):
    # One rounding from fp64, worked by hand; several cases differ from rounding
    # through fp32 first.
    for expr, h_hex, why in _golden("bf16_from_f64.json")["cases"]:
        v = float(eval(expr, {"__builtins__": {}}))
        got = int(o.bf16_from_f64(np.array([v]))[0])
        assert got == int(h_hex, 16), (expr, h_hex, hex(got), why)


def pin_bf16_vs_torch(o):
    import torch
    rng_bits = W.u64(5, 21, 4000).astype(np.uint32)
    vals = rng_bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    # Add ties and near-ties around random kept values.
    kept = (W.u64(6, 21, 500) & np.uint64(0x7F7F_0000)).astype(np.uint32)
    ties = np.concatenate([kept | 0x8000, kept | 0x7FFF, kept | 0x8001,
                           (kept | 0x1_0000) | 0x8000]).view(np.float32)
    vals = np.concatenate([vals, ties[np.isfinite(ties)]]).astype(np.float32)
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy()
    got = o.bf16_from_f32(vals).view(np.int16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Layout: counts, prefix sums, positions
# ---------------------------------------------------------------------------

def _layout_case(seed=1, T=37, N=41, E=16, K=3, R=4):
    ids = _ids(seed, T, E, K)
    return ids, N, E, K, R


def pin_counts_sum_and_bincount(o):
    for (T, N, E, K, R) in [(37, 41, 16, 3, 4), (64, 64, 8, 2, 2), (5, 8, 256, 8, 8),
                            (200, 203, 32, 4, 1)]:
        ids = _ids(T + E, T, E, K)
        lay = o.layout(ids, N, E, R)
        assert int(lay["cnt"].sum()) == T * K                      # sum of counts = T*K
        assert np.array_equal(lay["cnt"], np.bincount(ids.ravel(), minlength=E))
        assert int(lay["rank_prefix"][-1]) == T * K                # true total
        assert lay["err"] == 0


def pin_rank_totals_brute(o):
    ids, N, E, K, R = _layout_case(seed=3, T=29, N=31, E=12, K=4, R=3)
    T = ids.shape[0]
    lay = o.layout(ids, N, E, R)
    eloc = E // R
    rows = [0] * R
    toks = [0] * R
    for t in range(T):
        seen = set()
        for k in range(K):
            r = int(ids[t, k]) // eloc
            rows[r] += 1
            seen.add(r)
        for r in seen:
            toks[r] += 1
    assert lay["rows_per_rank"].tolist() == rows
    assert lay["tokens_in_rank"].tolist() == toks
    run, pre = 0, []
    for r in range(R):
        run += rows[r]
        pre.append(run)
    assert lay["rank_prefix"].tolist() == pre


def pin_positions_stable_sort(o):
    # Independent formulation: numpy's stable argsort of the flat pairs by
    # expert id gives the receive order; the j-th pair of rank r sits at r*S + j.
    for (seed, T, N, E, K, R) in [(4, 37, 41, 16, 3, 4), (5, 100, 100, 8, 2, 2),
                                  (6, 13, 16, 256, 8, 8), (7, 300, 301, 64, 6, 8)]:
        ids = _ids(seed, T, E, K)
        lay = o.layout(ids, N, E, R)
        S = lay["S"]
        flat = ids.ravel().astype(np.int64)
        order = np.argsort(flat, kind="stable")
        ranks = flat[order] // (E // R)
        want = np.empty(T * K, np.int64)
        for r in range(R):
            sel = order[ranks == r]
            want[sel] = r * S + np.arange(sel.size)
        assert np.array_equal(lay["pos"].ravel().astype(np.int64), want)
        # expert offsets: first row of each non-empty expert
        for e in range(E):
            hits = lay["pos"].ravel()[flat == e]
            if hits.size:
                assert int(hits.min()) == int(lay["expert_offset"][e])


def pin_positions_bijection(o):
    ids, N, E, K, R = _layout_case(seed=8, T=61, N=64, E=32, K=5, R=4)
    lay = o.layout(ids, N, E, R)
    S = lay["S"]
    pos = lay["pos"].ravel()
    assert np.unique(pos).size == pos.size
    for r in range(R):
        mine = np.sort(pos[(pos >= r * S) & (pos < (r + 1) * S)])
        assert np.array_equal(mine, r * S + np.arange(lay["rows_per_rank"][r]))


def pin_stride_and_shift(o):
    # Extents depend only on (N, K): S = pad(N) * K, and changing N moves each
    # rank's rows by r * (S2 - S1) and nothing else.
    ids = _ids(9, 13, 16, 2)
    a = o.layout(ids, 13, 16, 4)
    b = o.layout(ids, 40, 16, 4)
    assert a["S"] == 16 * 2 and b["S"] == 40 * 2
    ra = a["pos"] // a["S"]
    assert np.array_equal(a["pos"] - ra * a["S"], b["pos"] - ra * b["S"])
    assert np.array_equal(a["cnt"], b["cnt"])


def pin_padded_rows_route_nowhere(o):
    # Padded rows [T, P) of the routing map are all-False with zero probability;
    # real rows carry exactly their K ids and scores.
    T, N, E, K = 13, 13, 8, 2
    ids = _ids(10, T, E, K)
    sc = W.topk_scores(10, ids, E, "softmax_all")
    m, pr, err = o.routing_map(ids, sc, N, E)
    assert m.shape == (16, E) and err == 0
    assert not m[T:].any() and not pr[T:].any()
    for t in range(T):
        assert sorted(np.nonzero(m[t])[0].tolist()) == sorted(ids[t].tolist())
        for k in range(K):
            assert pr[t, ids[t, k]] == sc[t, k]
    # and the layout never counts a padded row
    lay = o.layout(ids, N, E, 2)
    assert int(lay["cnt"].sum()) == T * K


def pin_bad_and_duplicate_ids(o):
    ids = np.array([[3, 3], [8, 1], [-1, 2], [-5, 0]], dtype=np.int32)   # E = 8
    lay = o.layout(ids, 4, 8, 2)
    assert lay["err"] & 1
    assert lay["pos"][1, 0] == -1 and lay["pos"][2, 0] == -1 and lay["pos"][3, 0] == -1
    assert int(lay["cnt"][3]) == 2 and int(lay["cnt"].sum()) == 5
    assert lay["pos"][0, 1] == lay["pos"][0, 0] + 1


def pin_empty_call(o):
    ids = np.zeros((0, 4), np.int32)
    lay = o.layout(ids, 0, 8, 2)
    assert lay["S"] == 0 and not lay["cnt"].any() and not lay["rank_prefix"].any()
    lay = o.layout(ids, 6, 8, 2)
    assert lay["S"] == 8 * 4 and not lay["rows_per_rank"].any()


# ---------------------------------------------------------------------------
# Dispatch and combine
# ---------------------------------------------------------------------------

def pin_dispatch_rows(o):
    T, N, E, K, R, D = 23, 26, 16, 3, 4, 8
    ids = _ids(11, T, E, K)
    x = W.normal(11, 1, T * D).astype(np.float32).reshape(T, D)
    sc = W.topk_scores(11, ids, E, "sigmoid_norm")
    d = o.dispatch(x, sc, ids, N, E, R)
    for t in range(T):
        for k in range(K):
            p = d["pos"][t, k]
            assert np.array_equal(d["recv_x"][p], x[t])
            assert d["recv_src"][p] == t * K + k
            assert d["recv_scores"][p] == sc[t, k]
    # rows past each rank's true total are untouched
    used = np.zeros(R * d["S"], bool)
    used[d["pos"].ravel()] = True
    assert np.all(d["recv_src"][~used] == -1)


def pin_combine_identity_exact(o):
    # Identity experts: combine(dispatch(x))[t] = sum_k s_k * x_t, exact here.
    T, N, E, K, R, D = 19, 20, 16, 4, 4, 24
    ids = _ids(12, T, E, K)
    x, sc = _exact_inputs(12, T, D, K)
    want = (sc.astype(np.float64).sum(axis=1)[:, None] * x.astype(np.float64))
    for kind in ("f32", "bf16"):
        xin = x if kind == "f32" else _bf16_bits(x)
        d = o.dispatch(xin, sc, ids, N, E, R)
        out, err = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R, "f32")
        assert err == 0
        assert np.array_equal(out.astype(np.float64), want)


def pin_combine_scaled_experts_exact(o):
    # Expert e scales its rows by 2^((e mod 4) - 1): out[t] = sum_k s_k 2^j(e_k) x_t.
    # Distinct per-expert scales catch a gather from the wrong row or k.
    T, N, E, K, R, D = 17, 17, 8, 3, 2, 16
    ids = _ids(13, T, E, K)
    x, sc = _exact_inputs(13, T, D, K)
    d = o.dispatch(x, sc, ids, N, E, R)
    y = d["recv_x"].copy()
    for t in range(T):
        for k in range(K):
            y[d["pos"][t, k]] *= np.float32(2.0 ** ((ids[t, k] % 4) - 1))
    out, err = o.combine(y, sc, d["pos"], d["rank_prefix"], d["S"], R, "f32")
    scale = 2.0 ** ((ids % 4) - 1)
    want = (sc.astype(np.float64) * scale).sum(axis=1)[:, None] * x.astype(np.float64)
    assert err == 0 and np.array_equal(out.astype(np.float64), want)


def pin_combine_error_bound(o):
    # General inputs: the fp32 chain of K fused multiply-adds is within
    # K * 2^-24 * sum_k |s_k y_k| of the exact sum (fp64 here), and its bf16
    # rounding equals torch's bf16 cast of the oracle's own fp32 value.
    import torch
    T, N, E, K, R, D = 31, 33, 32, 8, 8, 40
    ids = W.topk_ids_zipf(14, T, E, K)
    sc = W.topk_scores(14, ids, E, "sigmoid_norm")
    x = W.hidden(14, T, D, "bf16")
    d = o.dispatch(x, sc, ids, N, E, R)
    out32, _ = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R, "f32")
    outbf, _ = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R, "bf16")
    xf = _f32_from_bits(x).astype(np.float64)
    s64 = sc.astype(np.float64)
    exact = s64.sum(axis=1)[:, None] * xf
    mag = np.abs(s64).sum(axis=1)[:, None] * np.abs(xf)
    assert np.all(np.abs(out32 - exact) <= K * 2.0 ** -24 * mag + 1e-45)
    ref = torch.from_numpy(out32).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(outbf.view(np.int16), ref)


def pin_unequal_count_invariance(o):
    # The pages' functional test: with identity experts a token's combined
    # output depends only on its own routing, so a run padded to the group max
    # reproduces, bit for bit, the run of the same tokens at their own count
    # and each token dispatched alone. Combos 8&3, 6&6, 5&3, 13&7.
    E, K, R, D = 16, 4, 4, 32
    for a, b in [(8, 3), (6, 6), (5, 3), (13, 7)]:
        n_group = max(a, b)
        for T in (a, b):
            ids = _ids(100 + T, T, E, K)
            sc = W.topk_scores(100 + T, ids, E, "sigmoid_norm")
            x = W.hidden(100 + T, T, D, "bf16")
            outs = []
            for N in (T, n_group):
                d = o.dispatch(x, sc, ids, N, E, R)
                out, err = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
                assert err == 0
                outs.append(out)
            assert np.array_equal(outs[0], outs[1])
            for t in range(T):
                d1 = o.dispatch(x[t:t + 1], sc[t:t + 1], ids[t:t + 1], 1, E, R)
                o1, _ = o.combine(d1["recv_x"], sc[t:t + 1], d1["pos"], d1["rank_prefix"],
                                  d1["S"], R)
                assert np.array_equal(o1[0], outs[0][t])


def pin_combine_rejects_rows_past_total(o):
    # A row beyond its rank's true total (from the prefix sum) contributes
    # nothing and is reported.
    T, N, E, K, R, D = 4, 4, 4, 1, 2, 8
    ids = np.array([[0], [1], [2], [3]], np.int32)
    x, sc = _exact_inputs(15, T, D, K)
    d = o.dispatch(x, sc, ids, N, E, R)
    pos = d["pos"].copy()
    pos[0, 0] = d["rows_per_rank"][0]        # first garbage row of rank 0
    out, err = o.combine(d["recv_x"], sc, pos, d["rank_prefix"], d["S"], R, "f32")
    assert err & 2
    assert not out[0].any()
    assert np.array_equal(out[1:], (sc[1:] * x[1:]).astype(np.float32))


# ---------------------------------------------------------------------------
# Backward: adjoint identities, finite differences, invariance
# ---------------------------------------------------------------------------

def _exact_grad(seed, T, D):
    gi = (W.u64(seed, 13, T * D) % np.uint64(65)).astype(np.int64) - 32
    return (gi.astype(np.float32) / np.float32(4.0)).reshape(T, D)


def pin_combine_backward_adjoint(o):
    # combine is linear in y: <combine(y), g> = <y, combine_backward_y(g)>,
    # exact in fp64 for dyadic fp32 data.
    T, N, E, K, R, D = 21, 24, 16, 4, 4, 12
    ids = _ids(30, T, E, K)
    x, sc = _exact_inputs(30, T, D, K)
    g = _exact_grad(30, T, D)
    d = o.dispatch(x, sc, ids, N, E, R)
    out, _ = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R, "f32")
    gy, _, err = o.combine_backward(g, d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
    assert err == 0
    lhs = float((out.astype(np.float64) * g).sum())
    valid = np.zeros(R * d["S"], bool)
    valid[d["pos"].ravel()] = True
    rhs = float((d["recv_x"][valid].astype(np.float64) * gy[valid]).sum())
    assert lhs == rhs


def pin_combine_backward_scores_by_difference(o):
    # grad_scores[t][k] is the change of <out, g> per unit change of s[t][k],
    # measured with the forward combine (exact for dyadic data).
    T, N, E, K, R, D = 9, 12, 8, 3, 2, 16
    ids = _ids(31, T, E, K)
    x, sc = _exact_inputs(31, T, D, K)
    g = _exact_grad(31, T, D)
    d = o.dispatch(x, sc, ids, N, E, R)
    _, gs, _ = o.combine_backward(g, d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
    base, _ = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R, "f32")
    delta = np.float32(1.0 / 64.0)
    for t in range(T):
        for k in range(K):
            s2 = sc.copy()
            s2[t, k] += delta
            o2, _ = o.combine(d["recv_x"], s2, d["pos"], d["rank_prefix"], d["S"], R, "f32")
            diff = float(((o2.astype(np.float64) - base) * g).sum())
            assert diff == float(delta) * float(gs[t, k]), (t, k)


def pin_combine_backward_grad_y_rounding(o):
    # bf16 grad_y is the bf16 rounding (torch's cast) of the fp32 product s * g.
    import torch
    T, N, E, K, R, D = 11, 12, 8, 2, 2, 32
    ids = _ids(32, T, E, K)
    sc = W.topk_scores(32, ids, E, "sigmoid_norm")
    x = W.hidden(32, T, D, "bf16")
    g = W.hidden(33, T, D, "bf16")
    d = o.dispatch(x, sc, ids, N, E, R)
    gy, _, _ = o.combine_backward(g, d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
    gf = _f32_from_bits(g)
    for t in range(T):
        for k in range(K):
            want = torch.from_numpy((sc[t, k] * gf[t]).astype(np.float32)).to(torch.bfloat16)
            assert np.array_equal(gy[d["pos"][t, k]].view(np.int16),
                                  want.view(torch.int16).numpy())


def pin_dispatch_backward_adjoint(o):
    # dispatch is linear in x and in s: <dispatch(x), G> = <x, grad_x> and
    # <recv_scores, h> = <s, grad_scores>, exact for dyadic fp32 data.
    T, N, E, K, R, D = 19, 20, 16, 4, 4, 10
    ids = _ids(34, T, E, K)
    x, sc = _exact_inputs(34, T, D, K)
    d = o.dispatch(x, sc, ids, N, E, R)
    rows = R * d["S"]
    G = _exact_grad(35, rows, D)
    h = _exact_grad(36, rows, 1).ravel()
    gx, gs, err = o.dispatch_backward(G, h, d["pos"], d["rank_prefix"], d["S"], R)
    assert err == 0
    valid = np.zeros(rows, bool)
    valid[d["pos"].ravel()] = True
    lhs = float((d["recv_x"][valid].astype(np.float64) * G[valid]).sum())
    assert lhs == float((x.astype(np.float64) * gx).sum())
    lhs_s = float((d["recv_scores"][valid].astype(np.float64) * h[valid]).sum())
    assert lhs_s == float((sc.astype(np.float64) * gs).sum())


def pin_backward_unequal_count_invariance(o):
    # [align] "Testing": forward AND backward reproduce the equal-count run
    # bit for bit. Per-token gradients do not depend on N or on other tokens.
    E, K, R, D = 16, 4, 4, 32
    for a, b in [(8, 3), (5, 3), (13, 7)]:
        T = b
        ids = _ids(200 + T, T, E, K)
        sc = W.topk_scores(200 + T, ids, E, "sigmoid_norm")
        x = W.hidden(200 + T, T, D, "bf16")
        g = W.hidden(300 + T, T, D, "bf16")
        res = []
        for N in (T, max(a, b)):
            d = o.dispatch(x, sc, ids, N, E, R)
            gy, gs, _ = o.combine_backward(g, d["recv_x"], sc, d["pos"], d["rank_prefix"],
                                           d["S"], R)
            gx, _, _ = o.dispatch_backward(gy, None, d["pos"], d["rank_prefix"], d["S"], R)
            res.append((gs, gx))
        assert np.array_equal(res[0][0].view(np.uint32), res[1][0].view(np.uint32))
        assert np.array_equal(res[0][1], res[1][1])


# ---------------------------------------------------------------------------
# Packed (exact-mode) layout
# ---------------------------------------------------------------------------

def pin_packed_positions_global_sort(o):
    # Packed rows: the j-th pair of numpy's stable argsort by expert sits at row j;
    # the rows fill exactly [0, true total).
    for (seed, T, N, E, K, R) in [(50, 37, 41, 16, 3, 4), (51, 13, 16, 256, 8, 8),
                                  (52, 120, 123, 32, 4, 1)]:
        ids = _ids(seed, T, E, K)
        lay = o.layout(ids, N, E, R, packed=True)
        order = np.argsort(ids.ravel(), kind="stable")
        want = np.empty(T * K, np.int64)
        want[order] = np.arange(T * K)
        assert np.array_equal(lay["pos"].ravel().astype(np.int64), want)
        assert int(lay["rank_prefix"][-1]) == T * K


def pin_packed_relation_to_strided(o):
    # The packed row of a pair is its strided row moved from r*S to the start
    # of rank r's rows in the packed buffer (the exclusive rank prefix).
    ids = _ids(53, 29, 16, 4)
    st = o.layout(ids, 31, 16, 4)
    pk = o.layout(ids, 31, 16, 4, packed=True)
    r = st["pos"] // st["S"]
    start = np.concatenate([[0], st["rank_prefix"][:-1]])[r]
    assert np.array_equal(pk["pos"], st["pos"] - r * st["S"] + start)


def pin_packed_combine_and_backward_match_strided(o):
    T, N, E, K, R, D = 23, 24, 16, 4, 4, 16
    ids = _ids(54, T, E, K)
    sc = W.topk_scores(54, ids, E, "sigmoid_norm")
    x = W.hidden(54, T, D, "bf16")
    g = W.hidden(55, T, D, "bf16")
    res = []
    for packed in (False, True):
        d = o.dispatch(x, sc, ids, N, E, R, packed=packed)
        out, err = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R,
                             packed=packed)
        gy, gs, _ = o.combine_backward(g, d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"],
                                       R, packed=packed)
        gx, _, _ = o.dispatch_backward(gy, None, d["pos"], d["rank_prefix"], d["S"], R,
                                       packed=packed)
        assert err == 0
        res.append((out, gs, gx))
    for a, b in zip(*res):
        assert np.array_equal(a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32),
                              b.view(np.uint16) if b.dtype == np.uint16 else b.view(np.uint32))


# ---------------------------------------------------------------------------
# Expert consumer (grouped GEMM)
# ---------------------------------------------------------------------------

def _gemm_case(seed=60, T=29, N=32, E=8, K=2, R=2, din=32, dout=24):
    ids = _ids(seed, T, E, K)
    sc = W.topk_scores(seed, ids, E, "sigmoid_norm")
    x = W.hidden(seed, T, din, "bf16")
    return ids, sc, x, N, E, K, R, din, dout


def _bf16_once(a64):
    """fp64 values rounded once to bf16 (8 significant bits, nearest, ties to
    even) by mpmath's correctly rounded conversion; the values here are normal
    in bf16, so its unbounded exponent does not matter."""
    import mpmath.libmp as L
    out = np.empty(a64.size, np.uint16)
    for i, v in enumerate(np.asarray(a64, np.float64).ravel()):
        r = np.float32(L.to_float(L.from_float(float(v), 8, "n")))
        out[i] = int(np.array([r]).view(np.uint32)[0]) >> 16
    return out.reshape(np.shape(a64))


def pin_expert_gemm_vs_numpy(o):
    # Each expert's rows times its weights, against numpy's fp64 matmul of the
    # same bf16 values, rounded once to bf16 by mpmath.
    ids, sc, x, N, E, K, R, din, dout = _gemm_case()
    d = o.dispatch(x, sc, ids, N, E, R)
    w = W.hidden(61, E * dout, din, "bf16").reshape(E, dout, din)
    y = o.expert_gemm(d["recv_x"], w, d["cnt"], d["expert_offset"], fill=0xFFFF)
    xf = _f32_from_bits(d["recv_x"]).astype(np.float64)
    wf = _f32_from_bits(w).astype(np.float64)
    covered = np.zeros(y.shape[0], bool)
    for e in range(E):
        lo, n = int(d["expert_offset"][e]), int(d["cnt"][e])
        ref = xf[lo:lo + n] @ wf[e].T
        assert np.array_equal(y[lo:lo + n], _bf16_once(ref))
        covered[lo:lo + n] = True
    assert np.all(y[~covered] == 0xFFFF)              # rows of no expert untouched


def pin_expert_gemm_single_rounding(o):
    # x = (1, 2^-8, 2^-30, 0...) against unit weights: the exact sum 1 + 2^-8 +
    # 2^-30 lies just above the bf16 tie at 1 + 2^-8, so one rounding gives
    # 1 + 2^-7 (3f81); rounding through fp32 first loses the 2^-30 and the tie
    # goes to even (3f80).
    E, K, R, din, dout, T = 2, 1, 1, 16, 16, 4
    ids = np.zeros((T, K), np.int32)
    sc = np.ones((T, K), np.float32)
    x = np.zeros((T, din), np.float32)
    x[:, 0], x[:, 1], x[:, 2] = 1.0, 2.0 ** -8, 2.0 ** -30
    d = o.dispatch(_bf16_bits(x), sc, ids, T, E, R)
    w = np.broadcast_to(_bf16_bits(np.ones((dout, din), np.float32)), (E, dout, din)).copy()
    y = o.expert_gemm(d["recv_x"], w, d["cnt"], d["expert_offset"])
    assert np.all(y[d["pos"].ravel()] == 0x3F81), hex(int(y[0, 0]))


def pin_expert_gemm_identity_weights(o):
    # W_e = [I | 0] (dout <= din): every expert copies the first dout columns.
    ids, sc, x, N, E, K, R, din, dout = _gemm_case(seed=62, din=32, dout=16)
    d = o.dispatch(x, sc, ids, N, E, R)
    eye = np.zeros((dout, din), np.float32)
    eye[np.arange(dout), np.arange(dout)] = 1.0
    w = np.broadcast_to(_bf16_bits(eye), (E, dout, din)).copy()
    y = o.expert_gemm(d["recv_x"], w, d["cnt"], d["expert_offset"])
    rows = d["pos"].ravel()
    assert np.array_equal(y[rows], d["recv_x"][rows, :dout])


# ---------------------------------------------------------------------------
# Per-rank dedupe
# ---------------------------------------------------------------------------

def pin_dedup_rows_brute(o):
    # Rank r's rows are exactly the tokens with an expert on r, in token order;
    # their count is the layout's tokens_in_rank; idx/w follow the pairs.
    T, N, E, K, R, D = 31, 33, 16, 4, 4, 8
    ids = _ids(70, T, E, K)
    sc = W.topk_scores(70, ids, E, "sigmoid_norm")
    x = W.hidden(70, T, D, "bf16")
    dd = o.dispatch_dedup(x, sc, ids, N, E, R)
    lay = o.layout(ids, N, E, R)
    assert np.array_equal(dd["tokens_in_rank"], lay["tokens_in_rank"])
    P, eloc = dd["P"], E // R
    for r in range(R):
        toks = [t for t in range(T) if any(int(e) // eloc == r for e in ids[t])]
        rows = np.arange(r * P, r * P + len(toks))
        assert dd["recv_tok_src"][rows].tolist() == toks
        for q, t in zip(rows, toks):
            assert np.array_equal(dd["recv_tok_x"][q], x[t])
            assert dd["tok_pos"][t, r] == q
            for k in range(K):
                e = int(ids[t, k])
                mine = e // eloc == r
                assert dd["recv_topk_idx"][q, k] == (e - r * eloc if mine else -1)
                assert dd["recv_topk_w"][q, k] == (sc[t, k] if mine else 0.0)
        others = [t for t in range(T) if t not in toks]
        assert all(dd["tok_pos"][t, r] == -1 for t in others)


def pin_dedup_expand_reproduces_dispatch(o):
    # The receiver's expansion of the dedupe rows equals the per-expert
    # dispatch bit for bit on every routed row.
    T, N, E, K, R, D = 45, 48, 32, 8, 8, 16
    ids = W.topk_ids_zipf(71, T, E, K)
    sc = W.topk_scores(71, ids, E, "sigmoid_norm")
    x = W.hidden(71, T, D, "bf16")
    d = o.dispatch(x, sc, ids, N, E, R)
    dd = o.dispatch_dedup(x, sc, ids, N, E, R)
    y = o.dedup_expand(dd["recv_tok_x"], dd["tok_pos"], d["pos"], ids, E, R, R * d["S"])
    rows = d["pos"].ravel()
    assert np.array_equal(y[rows], d["recv_x"][rows])
    assert int(dd["tokens_in_rank"].sum()) < T * K           # duplicates were folded


# ---------------------------------------------------------------------------
# Summation order and precision, by inputs where they change the exact result
# ---------------------------------------------------------------------------

def pin_combine_ascending_k_fma_chain(o):
    # One token, K = 3, y rows of ones, scores (1, 2^-24, -1). The fp32 chain in
    # ascending k: fma(1,1,0) = 1; fma(2^-24,1,1) = 1 + 2^-24, a tie that rounds
    # to even, 1; fma(-1,1,1) = 0. Descending k would give 2^-24 instead.
    T, N, E, K, R, D = 1, 1, 4, 3, 1, 4
    for ids in (np.array([[0, 1, 2]], np.int32), np.array([[2, 0, 1]], np.int32)):
        x = np.ones((T, D), np.float32)
        sc = np.array([[1.0, 2.0 ** -24, -1.0]], np.float32)
        d = o.dispatch(x, sc, ids, N, E, R)
        out, err = o.combine(d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R, "f32")
        assert err == 0
        assert np.array_equal(out.view(np.uint32), np.zeros((T, D), np.uint32))


def pin_expert_gemm_exact_cancellation(o):
    # x row (2^24, thirty-two ones, -2^24) against a weight row of ones: the exact
    # dot product is 32, which bf16 holds; a running fp32 sum loses every 1
    # against 2^24 (its spacing there is 2) and would return 0.
    din, dout, E = 34, 2, 1
    row = np.concatenate([[2.0 ** 24], np.ones(32), [-(2.0 ** 24)]]).astype(np.float32)
    x = _bf16_bits(row[None, :])
    w = _bf16_bits(np.ones((E * dout, din), np.float32)).reshape(E, dout, din)
    y = o.expert_gemm(x, w, np.array([1], np.int32), np.array([0], np.int32))
    assert np.array_equal(_f32_from_bits(y), np.full((1, dout), 32.0, np.float32))


def pin_combine_backward_score_gradient_exact(o):
    # grad_scores[t][k] = <grad_out[t], y[pos[t][k]]>, summed exactly and rounded
    # once: grad_out (2^24, thirty-two ones, -2^24) against a row of ones is 32;
    # a running fp32 sum would give 0.
    T, N, E, K, R = 1, 1, 2, 1, 1
    D = 34
    x = np.ones((T, D), np.float32)
    ids = np.array([[1]], np.int32)
    sc = np.array([[0.5]], np.float32)
    g = np.concatenate([[2.0 ** 24], np.ones(32), [-(2.0 ** 24)]]).astype(np.float32)[None, :]
    d = o.dispatch(x, sc, ids, N, E, R)
    _, gs, err = o.combine_backward(g, d["recv_x"], sc, d["pos"], d["rank_prefix"], d["S"], R)
    assert err == 0
    assert gs[0, 0] == np.float32(32.0)


# ---------------------------------------------------------------------------
# IEEE special values: overflow, signed zero, infinities, NaN, subnormals
# ---------------------------------------------------------------------------

def pin_bf16_nan_stays_nan(o):
    # A NaN must round to a NaN of the same sign, even when all of its payload
    # sits in the dropped low half (truncation would turn 7f800001 into +inf).
    for f_hex in ("7fc00000", "7f800001", "ff800001", "7fffffff", "ffc00000", "7f80ffff"):
        f = np.array([int(f_hex, 16)], dtype=np.uint32).view(np.float32)
        h = int(o.bf16_from_f32(f)[0])
        assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0, (f_hex, hex(h))
        assert (h >> 15) == (int(f_hex, 16) >> 31), (f_hex, hex(h))


BF16_MAX, BF16_MIN_SUB = 0x7F7F, 0x0001
NAN_BF16, NAN_F32 = 0x7FC0, 0x7FC00000      # the canonical quiet NaN


def special_value_case():
    """Six tokens, two experts each (ids [0, 1], one rank), and the two rows
    each token gathers, every element of a row the same bf16 value. Returns
    (ids, scores, rows [T, 2] of bf16 patterns, expected bf16 output per
    token, None where the result is NaN). The expected values follow from the
    fma chain acc = fma(s1, y1, fma(s0, y0, +0)) and round-to-nearest-even:
      0: max + 2^119 = (2 - 2^-8) 2^127 exactly, a tie above the largest
         finite bf16 with an odd kept bit: +inf;
      1: max + 2^118 = (2 - 2^-7 + 2^-9) 2^127, below the tie: max;
      2: -0 + -0 from an accumulator of +0: fma(1, -0, +0) = +0, so +0;
      3: +inf + -inf: NaN;
      4: 0.75 * 2^-133 = 3 * 2^-135, an fp32 subnormal (0x0000c000), above
         the bf16 tie: the smallest bf16 subnormal, 0x0001 (a flush to zero
         would give 0);
      5: 0 * inf: NaN;
      6: a negative quiet NaN with a payload (ffd5) plus 1: NaN;
      7: a signalling NaN (7f81) plus 1: NaN.
    Every NaN result of the arithmetic is the canonical quiet NaN, 7fc0 in
    bf16 (7fc00000 in fp32), whatever NaN the operands or the hardware carry:
    IEEE 754-2008 6.2 fixes only that the result is a quiet NaN, so the one
    encoding is the reading taken; NaN_BF16 marks those tokens."""
    ids = np.tile(np.array([[0, 1]], np.int32), (8, 1))
    sc = np.array([[1, 1], [1, 1], [1, 1], [1, 1], [0.75, 0], [0, 1], [1, 1], [1, 1]],
                  np.float32)
    rows = np.array([[BF16_MAX, 0x7B00],        # max, 2^119
                     [BF16_MAX, 0x7A80],        # max, 2^118
                     [0x8000, 0x8000],          # -0, -0
                     [0x7F80, 0xFF80],          # +inf, -inf
                     [BF16_MIN_SUB, 0x3F80],    # 2^-133, 1 (weight 0)
                     [0x7F80, 0x3F80],          # +inf (weight 0), 1
                     [0xFFD5, 0x3F80],          # -NaN with payload, 1
                     [0x7F81, 0x3F80]],         # signalling NaN, 1
                    np.uint16)
    want = [0x7F80, BF16_MAX, 0x0000, NAN_BF16, BF16_MIN_SUB, NAN_BF16, NAN_BF16, NAN_BF16]
    return ids, sc, rows, want


def special_value_y(d, rows, D):
    """The receive buffer of dispatch result d with each token's two gathered
    rows replaced by the case's constant rows."""
    y = np.array(d["recv_x"], copy=True)
    for t in range(rows.shape[0]):
        for k in range(2):
            y[int(d["pos"][t, k])] = np.full(D, rows[t, k], np.uint16)
    return y


def bf16_is_nan(h):
    h = np.asarray(h, np.uint16)
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


def pin_combine_ieee_special_values(o):
    ids, sc, rows, want = special_value_case()
    T, D, E, R = ids.shape[0], 8, 2, 1
    x = np.zeros((T, D), np.uint16)
    d = o.dispatch(x, sc, ids, T, E, R)
    y = special_value_y(d, rows, D)
    out, err = o.combine(y, sc, d["pos"], d["rank_prefix"], d["S"], R)
    assert err == 0
    for t, w in enumerate(want):
        assert np.all(out[t] == w), (t, hex(int(out[t, 0])), hex(w))
    out32, _ = o.combine(y, sc, d["pos"], d["rank_prefix"], d["S"], R, "f32")
    assert np.array_equal(out32.view(np.uint32), special_value_f32(want, D))


def special_value_f32(want, D):
    """The fp32 combine outputs of special_value_case: token 0 keeps the exact
    sum (2 - 2^-8) 2^127 = 0x7f7f8000, token 1 max + 2^118 = 0x7f7f4000, token 2
    +0, token 4 the subnormal 0x0000c000, the NaN tokens 0x7fc00000."""
    f32 = {0: 0x7F7F8000, 1: 0x7F7F4000, 2: 0x00000000, 4: 0x0000C000}
    rows = [NAN_F32 if w == NAN_BF16 else f32[t] for t, w in enumerate(want)]
    return np.repeat(np.array(rows, np.uint32)[:, None], D, axis=1)


def pin_backward_nan_canonical(o):
    # The backward's NaN results (s * NaN in grad_y, a NaN in grad_x's sum) are
    # the canonical quiet NaN however the incoming NaN is encoded (negative,
    # signalling, with a payload); finite entries are untouched.
    T, N, E, K, R, D = 6, 8, 4, 2, 2, 8
    ids = np.array([[0, 2], [1, 3], [0, 1], [2, 3], [3, 0], [1, 2]], np.int32)
    sc = np.full((T, K), 0.5, np.float32)
    x = _bf16_bits(np.ones((T, D), np.float32))
    d = o.dispatch(x, sc, ids, N, E, R)
    g = _bf16_bits(np.ones((T, D), np.float32))
    g[0, :] = 0xFFD5        # negative quiet NaN with a payload
    g[1, :4] = 0x7F81       # signalling NaN
    g[2, 0] = 0x7FEA        # quiet NaN with a payload
    for kind, nan in (("bf16", NAN_BF16), ("f32", NAN_F32)):
        gk = g if kind == "bf16" else _f32_from_bits(g)
        yk = d["recv_x"] if kind == "bf16" else _f32_from_bits(d["recv_x"])
        gy, _, _ = o.combine_backward(gk, yk, sc, d["pos"], d["rank_prefix"], d["S"], R)
        gy_bits = gy.view(np.uint16 if kind == "bf16" else np.uint32)
        half = 0x3F00 if kind == "bf16" else 0x3F000000
        gx, _, _ = o.dispatch_backward(gy, None, d["pos"], d["rank_prefix"], d["S"], R)
        gx_bits = gx.view(np.uint16 if kind == "bf16" else np.uint32)
        one = 0x3F80 if kind == "bf16" else 0x3F800000
        nan_in = bf16_is_nan(g)
        for t in range(T):
            for k in range(K):
                row = gy_bits[d["pos"][t, k]]
                assert np.array_equal(row, np.where(nan_in[t], nan, half)), (kind, t, k)
            assert np.array_equal(gx_bits[t], np.where(nan_in[t], nan, one)), (kind, t)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
