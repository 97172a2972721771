"""The one-pass dispatch's token pool, as host arithmetic: every token of a
call is copied exactly once, whether by its own tile or from the pool.

Tile c holds tokens [c*tpt, min(T, (c+1)*tpt)); of its n tokens it keeps the
first n - share(n) (at least a ring of `stages` rows, loaded before the layout
is known) and gives the last share(n) = min(d, max(0, n - stages)) to the pool,
where d = min(tpt * pct / 100, tpt - stages). Pool entry e (taken in order from
one shared counter) is token e // ntiles of tile e % ntiles's share, or nothing
if that share is shorter. This restates the kernel's mapping (permute.cu) so
that a change to it is checked on every shape class: full and short last tiles,
tiles that fit the ring (no pool), shares of zero, of some and of all but a
ring's worth.
"""
import itertools


def tiling(T, tpt):
    ntiles = (T + tpt - 1) // tpt
    return ntiles, [min(T, (c + 1) * tpt) - c * tpt for c in range(ntiles)]


def pool_depth(tpt, stages, pct):
    return max(0, min(tpt * pct // 100, tpt - stages))


def copied_tokens(T, tpt, stages, d):
    ntiles, sizes = tiling(T, tpt)
    share = [min(d, max(0, n - stages)) for n in sizes]
    got = []
    for c, n in enumerate(sizes):            # each tile's own tokens
        got += [c * tpt + q for q in range(n - share[c])]
    for e in range(ntiles * d):              # the pool, in counter order
        c, j = e % ntiles, e // ntiles
        if j < share[c]:
            got.append(c * tpt + (sizes[c] - share[c]) + j)
    return got


def test_every_token_once():
    cases = 0
    for T, tpt in itertools.product([1, 2, 3, 7, 16, 40, 151, 152, 153, 1000, 4096, 8192],
                                    [1, 2, 3, 5, 12, 27, 54]):
        if tpt > T:
            continue
        for stages, pct in itertools.product((6, 15, 26, 32), (0, 10, 25, 50, 100)):
            d = pool_depth(tpt, stages, pct)
            got = copied_tokens(T, tpt, stages, d)
            assert sorted(got) == list(range(T)), (T, tpt, stages, d)
            cases += 1
    assert cases >= 1000


def test_pool_entries_mostly_full():
    # Only the short last tile can leave pool entries empty (at most d of them),
    # so CTAs do not spend their atomics on empty entries; tiles that fit the
    # ring have no pool at all (d = 0).
    for T, tpt, stages, pct, want_d in [(4096, 27, 26, 25, 1), (8192, 54, 15, 25, 13),
                                        (1792, 12, 15, 25, 0), (32768, 216, 15, 25, 54)]:
        d = pool_depth(tpt, stages, pct)
        assert d == want_d
        ntiles, sizes = tiling(T, tpt)
        share = [min(d, max(0, n - stages)) for n in sizes]
        assert sum(d - s for s in share) <= d
