"""A CPU model of how the recurrence kernel splits the work and sums the
carries, checked for exact coverage: every group's partial sum of a row is
counted once in that row's total (in part B or in the carry a CTA publishes
for the row it ends inside), on the FlyGPT-shaped graph and on random graphs,
for row-weighted merge-path pieces of several weights.

The model follows the kernel's rules: piece c starts at diagonal
(E + w N) S(c) / S(P), where S(c) sums the shares of pieces [0, c): 1000 + L
per mille for the first half, 1000 - L for the second (the graph build's
late-dispatch share L), so L = 0 is the even cut c (E + w N) / P (rows whose
ends come first, edges between their row pointers); lane group g of G takes edges [e0 + g n / G, e0 + (g+1) n / G); a
group's carry belongs to the row of its last edge (an empty group takes the
row of edge k0); groups of a warp (EPW of them) with the same row add their
carries by a segmented suffix sum, so a row spanning groups [ga, gb) reads
group ga and the first group of every later warp below gb.  Integer carries
make the sums exact.
"""
import numpy as np

import workloads


def _piece(row_ptr, N, w, d):
    lo, hi = 0, N
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if row_ptr[mid] + w * mid <= d:
            lo = mid
        else:
            hi = mid - 1
    return lo, min(d - w * lo, row_ptr[min(lo + 1, N)])


def _share_prefix(c, P, late):
    h = P // 2
    return c * (1000 + late) if c <= h else h * (1000 + late) + (c - h) * (1000 - late)


def _diagonal(c, P, items, late):
    return items if c == P else items * _share_prefix(c, P, late) // _share_prefix(P, P, late)


def _check(row_ptr, N, E, P, G, EPW, w, rng, late=15):
    items = E + w * N
    rowid = np.repeat(np.arange(N), np.diff(row_ptr))
    for cta in range(P):
        (r0, e0) = _piece(row_ptr, N, w, _diagonal(cta, P, items, late))
        (r1, e1) = _piece(row_ptr, N, w, _diagonal(cta + 1, P, items, late))
        n, nrows = e1 - e0, r1 - r0
        assert row_ptr[r0] <= e0 <= e1 and nrows >= 0
        carry = np.zeros(G, np.int64)
        lab = np.full(G, -1)
        truth = {}
        for g in range(G):
            k0 = e0 + (g * n // G if n else 0)
            k1 = e0 + ((g + 1) * n // G if n else 0)
            if k1 > k0:
                cur = rowid[k1 - 1]
                fin = r0 <= cur < r0 + nrows and row_ptr[cur + 1] == k1
                v = 0 if fin else int(rng.integers(1, 1000))
                carry[g], lab[g] = v, cur
                if v:
                    truth[cur] = truth.get(cur, 0) + v
            else:
                lab[g] = rowid[k0] if k0 < e1 else -1
        s = carry.copy()
        d = 1
        while d < EPW:
            nxt = s.copy()
            for g in range(G):
                if g % EPW + d < EPW and lab[g + d] == lab[g]:
                    nxt[g] += s[g + d]
            s, d = nxt, d * 2

        def group_of(k):
            return min(((k - e0 + 1) * G - 1) // n, G - 1)

        def heads(ga, gb):
            hs = [ga] if ga < gb else []
            h = (ga // EPW + 1) * EPW
            while h < gb:
                hs.append(h)
                h += EPW
            return hs

        got = {}
        for r in range(r0, r1):
            rs, re = row_ptr[r], row_ptr[r + 1]
            if re > rs and re - 1 >= e0:
                got[r] = sum(int(s[h]) for h in heads(group_of(max(rs, e0)), group_of(re - 1)))
        if r1 < N and cta + 1 < P and n > 0:
            ka = max(row_ptr[r1], e0)
            ga = group_of(ka) if ka < e1 else G
            got[r1] = got.get(r1, 0) + sum(int(s[h]) for h in heads(ga, G))
        for r in set(truth) | set(got):
            assert got.get(r, 0) == truth.get(r, 0), (cta, r)


def test_flygpt_pieces_and_carries():
    rng = np.random.default_rng(0)
    c = workloads.make(1, with_dout=False)
    N = c["N"]
    for key in ("dst", "src"):
        rp = np.zeros(N + 1, np.int64)
        np.add.at(rp, np.asarray(c[key]) + 1, 1)
        rp = np.cumsum(rp)
        # two CTAs of 8 warps per SM (304 pieces, 64 groups of 4 lanes each)
        # and one CTA of 16 warps (152 pieces, 128 groups); the row weights
        # the cost model picks for this graph (16 forward, 1 backward) and 3
        for P, G in ((304, 64), (152, 128)):
            for w in (1, 3, 16):
                for late in (0, 15):
                    _check(rp, N, int(rp[-1]), P, G, 8, w, rng, late)


def test_random_graphs_pieces_and_carries():
    rng = np.random.default_rng(1)
    for _ in range(120):
        N = int(rng.integers(1, 300))
        E = int(rng.integers(0, 2500))
        P = int(rng.integers(1, 20))
        EPW = int(rng.choice([1, 2, 4, 8, 16, 32]))
        G = EPW * int(rng.integers(1, 5))
        deg = rng.multinomial(E, rng.dirichlet(np.ones(N) * rng.choice([0.05, 1.0])))
        rp = np.concatenate([[0], np.cumsum(deg)])
        _check(rp, N, E, P, G, EPW, int(rng.choice([1, 2, 3, 4, 8, 16])), rng,
               int(rng.choice([0, 15, 400])))


def test_late_share_cut():
    """The shares: the second half's pieces carry (1000 - L) / (1000 + L) of the
    first half's weighted items (to rounding), the diagonals rise and end at
    the total."""
    items, P, late = 604_324, 304, 15
    d = [_diagonal(c, P, items, late) for c in range(P + 1)]
    assert d[0] == 0 and d[-1] == items and all(a <= b for a, b in zip(d, d[1:]))
    first = np.diff(d[: P // 2 + 1]).mean()
    second = np.diff(d[P // 2:]).mean()
    assert abs(second / first - 985 / 1015) < 1e-4
