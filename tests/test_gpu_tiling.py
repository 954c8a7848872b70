"""The shared-memory tiling the graph build makes for the tiled kernels,
checked bit for bit against the oracle's compressed rows.

For each direction (rows keyed by dst; by src) the column nodes are cut into C
chunks and the rows into G blocks, and CTA t = g * C + j owns cell (g, j): the
edges of block g's rows whose column lies in chunk j, in row order and, within
a row, in the compressed-row order (ascending caller edge id).  Everything
here is integer work, so the test rebuilds every array from the oracle's
layout (oracle.graph_layout) and the chunk and block bounds the build chose,
and requires equality.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import make_graph

pytestmark = pytest.mark.gpu


def _export(g, d):
    from sparse_graph_recurrent_gb300 import _ck
    info = _ck.ck_graph_tiling(g.handle, d)
    if info["C"] == 0:
        return info, None
    E = int(g.E) if hasattr(g, "E") else None
    dev = torch.device("cuda")
    meta = torch.empty(info["P"] * 12, dtype=torch.int32, device=dev)
    ptr = torch.empty(max(info["ptr_len"], 1), dtype=torch.int32, device=dev)
    n_e = max(E, 1)
    col, perm, rowid = (torch.empty(n_e, dtype=torch.int32, device=dev) for _ in range(3))
    _ck.ck_graph_export_tiling(g.handle, d, meta, ptr, col, perm, rowid)
    torch.cuda.synchronize()
    arr = lambda t: t.cpu().numpy().astype(np.int64)  # noqa: E731
    return info, dict(meta=arr(meta).reshape(info["P"], 12), ptr=arr(ptr), col=arr(col)[:E],
                      perm=arr(perm)[:E], rowid=arr(rowid)[:E])


def _check_direction(c, info, t, d):
    N, E = c["N"], c["E"]
    lay = oracle.graph_layout(N, c["src"], c["dst"], c["input_nodes"])
    rp, col, perm = ((lay["row_ptr"], lay["col"], lay["perm"]) if d == 0 else
                     (lay["rowT_ptr"], lay["colT"], lay["permT"]))
    rp, col, perm = rp.astype(np.int64), col.astype(np.int64), perm.astype(np.int64)
    C, G, P = info["C"], info["G"], info["P"]
    assert P == G * C and P <= torch.cuda.get_device_properties(0).multi_processor_count
    m = t["meta"]
    # blocks: contiguous, in order, covering [0, N); chunks likewise
    blocks = [(m[gg * C, 0], m[gg * C, 1]) for gg in range(G)]
    assert blocks[0][0] == 0 and sum(r for _, r in blocks) == N
    for (r0, R), (r1, _) in zip(blocks, blocks[1:]):
        assert r0 + R == r1
    chunks = [(m[j, 4], m[j, 5]) for j in range(C)]
    assert chunks[0][0] == 0 and sum(n for _, n in chunks) == N
    chunk_of = np.empty(N, np.int64)
    for j, (c0, cn) in enumerate(chunks):
        chunk_of[c0:c0 + cn] = j
    seen = np.zeros(E, np.int64)
    rows = np.repeat(np.arange(N), np.diff(rp))
    in_chunk = chunk_of[col] if E else np.zeros(0, np.int64)
    pos = 0
    for tt in range(P):
        gg, j = tt // C, tt % C
        r0, R, e0, e1, c0, cn, poff, f0, f1, mj, mg, _ = m[tt]
        assert (mj, mg) == (j, gg) and (r0, R) == blocks[gg] and (c0, cn) == chunks[j]
        assert (f0, f1) == (R * j // C, R * (j + 1) // C)
        assert e0 == pos
        # the cell, rebuilt: rows of the block in order, each row's edges whose
        # column lies in chunk j, in compressed-row order
        span = np.arange(rp[r0], rp[r0 + R])
        wk = span[in_chunk[span] == j]
        assert e1 - e0 == len(wk), (tt, e1 - e0, len(wk))
        np.testing.assert_array_equal(t["col"][e0:e1], col[wk] - c0 if len(wk) else [])
        np.testing.assert_array_equal(t["perm"][e0:e1], perm[wk] if len(wk) else [])
        np.testing.assert_array_equal(t["rowid"][e0:e1], rows[wk] if len(wk) else [])
        # row pointers: R + 1 positions, each row's count of chunk-j edges
        per_row = np.bincount(rows[wk] - r0, minlength=R) if len(wk) else np.zeros(R, np.int64)
        exp_ptr = e0 + np.concatenate([[0], np.cumsum(per_row)])
        np.testing.assert_array_equal(t["ptr"][poff:poff + R + 1], exp_ptr)
        if len(wk):
            seen[wk] += 1
        pos = e1
    assert pos == E and (seen == 1).all()
    assert info["max_rows"] == max(R for _, R in blocks)
    assert info["max_chunk"] == max(n for _, n in chunks)


CASES = [
    # seed, N, E, n_in, B, T, M, extra
    (801, 1, 0, 1, 1, 1, 1, {}),
    (802, 2, 3, 1, 3, 2, 2, {}),
    (803, 64, 900, 6, 20, 2, 2, dict(hub_deg=400)),
    (804, 700, 40000, 12, 20, 4, 2, dict(hub_deg=9000)),
    (805, 3000, 200000, 32, 32, 2, 2, dict(hub_deg=150000)),
]


@pytest.mark.parametrize("seed,N,E,n_in,B,T,M,extra", CASES, ids=[f"N{c[1]}_E{c[2]}" for c in CASES])
def test_tiling_matches_compressed_rows(seed, N, E, n_in, B, T, M, extra):
    c = workloads.small(seed, N, E, n_in, B, T, M, **extra)
    g = make_graph(c, tiling=True)
    g.E = c["E"]
    for d in (0, 1):
        info, t = _export(g, d)
        assert info["C"] > 0, (d, info)
        _check_direction(c, info, t, d)


@pytest.mark.slow
def test_tiling_flygpt_shape():
    c = workloads.make(1)
    g = make_graph(c, tiling=True)
    g.E = c["E"]
    for d in (0, 1):
        info, t = _export(g, d)
        assert info["C"] > 0, (d, info)
        _check_direction(c, info, t, d)


def test_no_tiling_for_the_wide_graph():
    """A graph whose state rows need more than eight CTAs' shared memory has
    no tiling (its calls run the L2-gather kernels)."""
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(806, 20000, 60000, 8, 4, 1, 1)
    g = make_graph(c, tiling=True)
    for d in (0, 1):
        assert _ck.ck_graph_tiling(g.handle, d)["C"] == 0


def test_tiling_is_built_only_on_request():
    """A graph holds tilings only when created with CK_GRAPH_TILING (three int32
    arrays per edge and direction, plus O(N) tables); without them the tiled
    option runs the L2-gather kernels, bit for bit what the option off gives."""
    from sparse_graph_recurrent_gb300 import _ck
    from gpu_helpers import run_gpu
    c = workloads.small(807, 700, 40000, 12, 20, 4, 2, hub_deg=9000)
    plain, tiled = make_graph(c, tiling=False), make_graph(c, tiling=True)
    for d in (0, 1):
        assert _ck.ck_graph_tiling(plain.handle, d)["C"] == 0
        assert _ck.ck_graph_tiling(tiled.handle, d)["C"] > 0
    dev_plain, _ = _ck.ck_graph_memory(plain.handle)
    dev_tiled, _ = _ck.ck_graph_memory(tiled.handle)
    assert dev_tiled - dev_plain >= 2 * 3 * 4 * c["E"]
    try:
        _ck.ck_set_option(_ck.OPT_TILED, 0)
        off_out, off = run_gpu(c, graph=plain)
        _ck.ck_set_option(_ck.OPT_TILED, 1)
        on_out, on = run_gpu(c, graph=plain)
    finally:
        _ck.ck_set_option(_ck.OPT_TILED, 0)
    np.testing.assert_array_equal(on_out, off_out)
    for k in off:
        np.testing.assert_array_equal(on[k], off[k])
