"""The seeded synthetic inputs have the documented shapes and structure
(sizes, degree caps, hubs, unique pairs, value ranges) and are reproducible."""
import numpy as np
import pytest

import workloads

SIZES = {0: (256, 4096, 16, 8, 8, 2), 1: (5000, 524324, 64, 32, 64, 2),
         2: (5000, 524324, 64, 20, 32, 2), 3: (20000, 2000000, 256, 256, 32, 2),
         4: (211577, 24678466, 1024, 32, 16, 2)}


def _indeg(c):
    return np.bincount(np.asarray(c["dst"]), minlength=c["N"])


def _common(c, cid):
    N, E, n_in, B, T, M = SIZES[cid]
    assert (c["N"], c["E"], c["n_in"], c["B"], c["T"], c["M"]) == (N, E, n_in, B, T, M)
    src, dst = np.asarray(c["src"]), np.asarray(c["dst"])
    assert src.shape == dst.shape == (E,) and c["w"].shape == (E,)
    assert src.min() >= 0 and src.max() < N and dst.min() >= 0 and dst.max() < N
    assert c["leak"].shape == c["bias"].shape == (N,)
    assert np.all((c["leak"] > 0) & (c["leak"] < 1))  # a sigmoid's range
    assert c["drives"].shape == (T, n_in, B) and c["state0"].shape == (B, N)
    inp = np.asarray(c["input_nodes"])
    assert inp.shape == (n_in,) and len(np.unique(inp)) == n_in and inp.min() >= 0 and inp.max() < N
    assert not np.all(np.diff(dst) >= 0)  # the caller's order is not the row order
    return src, dst


@pytest.mark.parametrize("cid", [0, 1, 2, 3])
def test_shapes_and_structure(cid):
    c = workloads.make(cid, with_dout=cid != 3)  # the wide dOut alone is 1.3 GB
    src, dst = _common(c, cid)
    if cid != 3:
        assert c["dout"].shape == (c["T"], c["B"], c["N"])
    d = _indeg(c)
    if cid == 0:
        assert np.all(src != dst)
        assert len(np.unique(src.astype(np.int64) * c["N"] + dst)) == c["E"]
    elif cid == 2:
        assert np.sum(d == 8192) == 50 and np.sort(d)[-51] <= 2000 and d.min() >= 1
    else:
        dmax = {1: 2000, 3: 20000}[cid]
        assert d.min() >= 1 and d.max() <= dmax and d.sum() == c["E"]
        assert d.max() > 20 * np.median(d)  # heavy-tailed


def test_connectome_shape():
    c = workloads.make(4, with_dout=False)
    _common(c, 4)
    d = _indeg(c)
    assert d.min() >= 1 and d.max() <= 20000
    pos = np.mean(np.asarray(c["w"]) > 0)
    assert abs(pos - 0.7) < 0.01  # signed weights, P(+) = 0.7


def test_reproducible():
    a, b = workloads.make(1), workloads.make(1)
    for k in ("src", "dst", "w", "leak", "bias", "drives", "state0", "dout", "input_nodes"):
        np.testing.assert_array_equal(np.asarray(a[k]), np.asarray(b[k]))
    c = workloads.make(2)
    assert not np.array_equal(np.asarray(a["w"]), np.asarray(c["w"]))
