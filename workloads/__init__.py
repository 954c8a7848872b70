"""Seeded synthetic inputs for the sparse-graph leaky-tanh recurrence.

This module only draws random numbers and index lists; it holds none of the
recurrence's arithmetic.  The same arrays feed both the CPU oracle and the CUDA
library, so the two sides are always compared on identical inputs.

Workloads (shapes from the connectome-kernels page, "Why" table, and the
soup-connectome page, "Status" table, for the connectome size):

  0 tiny        N=256, E=4,096 unique (src,dst) pairs, no self-loops, n_in=16,
                B=8, T=8, M=2
  1 flygpt      N=5,000, E=524,324, power-law in-degree (alpha=2.0, clip
                [1, 2,000]), uniform sources, n_in=64, B=32, T=64, M=2
  2 ragged      as 1, with 50 hub nodes forced to in-degree 8,192, B=20, T=32,
                M in {1, 2, 3}
  3 wide        N=20,000, E=2,000,000, alpha=2.2, n_in=256, B=256, T=32, M=2
  4 connectome  N=211,577, E=24,678,466, alpha=2.0, max in-degree 20,000,
                n_in=1,024, B=32, T=16, M=2, edge values with a fixed random
                sign (+1 with p=0.7)

Every array is returned in numpy: indices as int64, values as float32 (the
precision of the CUDA path; the oracle widens the same float32 values to fp64).
"""
from __future__ import annotations

import numpy as np

# Child streams are spawned in this fixed order from SeedSequence(1000 + id).
_STREAMS = ("perm", "deg", "src", "shuffle", "w", "sign", "leak", "bias",
            "drives", "state0", "dout")

CONFIGS = {
    0: dict(name="tiny", N=256, E=4096, n_in=16, B=8, T=8, M=2),
    1: dict(name="flygpt", N=5000, E=524324, n_in=64, B=32, T=64, M=2,
            alpha=2.0, dmax=2000),
    2: dict(name="ragged", N=5000, E=524324, n_in=64, B=20, T=32, M=2,
            alpha=2.0, dmax=2000, hubs=50, hub_deg=8192),
    3: dict(name="wide", N=20000, E=2000000, n_in=256, B=256, T=32, M=2,
            alpha=2.2, dmax=20000),
    4: dict(name="connectome", N=211577, E=24678466, n_in=1024, B=32, T=16,
            M=2, alpha=2.0, dmax=20000, signed=True),
}


def _streams(seed: int) -> dict:
    kids = np.random.default_rng(np.random.SeedSequence(seed)).spawn(len(_STREAMS))
    return dict(zip(_STREAMS, kids))


def powerlaw_degrees(rng_deg, N: int, E: int, alpha: float, dmax: int) -> np.ndarray:
    """In-degrees d_i >= 1, d_i <= dmax, sum exactly E, shaped like a power law.

    x_i = (1-u)^(-1/(alpha-1)) (Pareto); a scale s is bisected so that
    sum(clip(floor(s*x_i), 1, dmax)) is the largest value <= E; the remainder
    is then added one unit at a time to nodes in a seeded random order,
    skipping nodes already at dmax.
    """
    if E < N or E > N * dmax:
        raise ValueError("power-law degrees need N <= E <= N*dmax")
    u = rng_deg.random(N)
    x = (1.0 - u) ** (-1.0 / (alpha - 1.0))

    def total(s):
        return int(np.clip(np.floor(s * x), 1, dmax).sum())

    lo, hi = 0.0, 1.0
    while total(hi) <= E:
        hi *= 2.0
        if hi > 1e18:
            break
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if total(mid) <= E:
            lo = mid
        else:
            hi = mid
    d = np.clip(np.floor(lo * x), 1, dmax).astype(np.int64)
    rem = E - int(d.sum())
    order = rng_deg.permutation(N)
    while rem > 0:
        room = order[d[order] < dmax]
        if room.size == 0:
            raise ValueError("cannot reach E under dmax")
        take = room[:rem]
        d[take] += 1
        rem -= take.size
    assert int(d.sum()) == E
    return d


def _edges_from_degrees(rs, indeg: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    N = indeg.size
    E = int(indeg.sum())
    dst = np.repeat(np.arange(N, dtype=np.int64), indeg)
    src = rs["src"].integers(0, N, size=E, dtype=np.int64)
    order = rs["shuffle"].permutation(E)
    return src[order], dst[order]


def _unique_pairs(rs, N: int, E: int) -> tuple[np.ndarray, np.ndarray]:
    """E distinct (src,dst) pairs with src != dst, drawn uniformly."""
    seen = set()
    src = np.empty(E, np.int64)
    dst = np.empty(E, np.int64)
    k = 0
    rng = rs["src"]
    while k < E:
        s, d = (int(v) for v in rng.integers(0, N, size=2))
        if s == d or (s, d) in seen:
            continue
        seen.add((s, d))
        src[k], dst[k] = s, d
        k += 1
    order = rs["shuffle"].permutation(E)
    return src[order], dst[order]


def _values(rs, N, E, n_in, B, T, signed):
    f32 = np.float32
    scale = 1.0 / np.sqrt(max(E / N, 1.0))
    if signed:
        mag = np.abs(rs["w"].normal(0.0, scale, E))
        sign = np.where(rs["sign"].random(E) < 0.7, 1.0, -1.0)
        w = sign * mag
    else:
        w = rs["w"].normal(0.0, scale, E)
    leak = 1.0 / (1.0 + np.exp(-rs["leak"].normal(0.0, 1.0, N)))
    bias = rs["bias"].normal(0.0, 0.1, N)
    drives = rs["drives"].normal(0.0, 1.0, (T, n_in, B))
    state0 = rs["state0"].normal(0.0, 0.1, (B, N))
    return dict(w=w.astype(f32), leak=leak.astype(f32), bias=bias.astype(f32),
                drives=drives.astype(f32), state0=state0.astype(f32))


def make(config_id: int, M: int | None = None, with_dout: bool = True) -> dict:
    """Inputs of one workload: graph, parameters, drives, state0 and dOut."""
    c = CONFIGS[config_id]
    rs = _streams(1000 + config_id)
    N, E, n_in, B, T = c["N"], c["E"], c["n_in"], c["B"], c["T"]
    M = c["M"] if M is None else M
    perm = rs["perm"].permutation(N).astype(np.int64)
    input_nodes = perm[:n_in].copy()
    if config_id == 0:
        src, dst = _unique_pairs(rs, N, E)
    elif "hubs" in c:
        hubs = perm[64:64 + c["hubs"]]
        is_hub = np.zeros(N, bool)
        is_hub[hubs] = True
        rest = np.flatnonzero(~is_hub)
        e_rest = E - c["hubs"] * c["hub_deg"]
        indeg = np.zeros(N, np.int64)
        indeg[hubs] = c["hub_deg"]
        indeg[rest] = powerlaw_degrees(rs["deg"], rest.size, e_rest, c["alpha"], c["dmax"])
        src, dst = _edges_from_degrees(rs, indeg)
    else:
        indeg = powerlaw_degrees(rs["deg"], N, E, c["alpha"], c["dmax"])
        src, dst = _edges_from_degrees(rs, indeg)
    out = dict(name=c["name"], N=N, E=E, n_in=n_in, B=B, T=T, M=M,
               src=src, dst=dst, input_nodes=input_nodes)
    out.update(_values(rs, N, E, n_in, B, T, c.get("signed", False)))
    if with_dout:
        out["dout"] = rs["dout"].normal(0.0, 1.0, (T, B, N)).astype(np.float32)
    return out


def small(seed: int, N: int, E: int, n_in: int, B: int, T: int, M: int,
          self_loops: bool = True, dup_frac: float = 0.0, hub_deg: int = 0,
          w_scale: float | None = None, src_hub_deg: int = 0, loops_only: bool = False) -> dict:
    """A random small case: uniform edges, optional duplicates and one hub row.

    dup_frac of the edges repeat an earlier (src,dst) pair; a hub row, if
    asked for, takes hub_deg of the E edges into node N-1; a source hub,
    src_hub_deg of them out of node 0 (a hub row of the transposed rows);
    loops_only turns every edge into a self-loop at its source.  The last two
    draw nothing when unset, so the other cases are unchanged by them.
    """
    rs = _streams(seed)
    perm = rs["perm"].permutation(N).astype(np.int64)
    input_nodes = perm[:n_in].copy()
    rng = rs["src"]
    n_hub = min(hub_deg, E)
    n_shub = min(src_hub_deg, E - n_hub)
    n_dup = int(round(dup_frac * (E - n_hub - n_shub)))
    n_base = E - n_hub - n_shub - n_dup
    src = rng.integers(0, N, size=n_base, dtype=np.int64)
    dst = rng.integers(0, N, size=n_base, dtype=np.int64)
    if not self_loops:
        bad = src == dst
        dst[bad] = (dst[bad] + 1) % N
    if n_dup:
        pick = rng.integers(0, max(n_base, 1), size=n_dup) if n_base else np.zeros(n_dup, np.int64)
        src = np.concatenate([src, src[pick] if n_base else rng.integers(0, N, n_dup)])
        dst = np.concatenate([dst, dst[pick] if n_base else rng.integers(0, N, n_dup)])
    if n_hub:
        src = np.concatenate([src, rng.integers(0, N, size=n_hub, dtype=np.int64)])
        dst = np.concatenate([dst, np.full(n_hub, N - 1, np.int64)])
    if n_shub:
        src = np.concatenate([src, np.zeros(n_shub, np.int64)])
        dst = np.concatenate([dst, rng.integers(0, N, size=n_shub, dtype=np.int64)])
    if loops_only:
        dst = src.copy()
    order = rs["shuffle"].permutation(E)
    src, dst = src[order].astype(np.int64), dst[order].astype(np.int64)
    mean_deg = max(E / N, 1.0)
    vals = _values(rs, N, E, n_in, B, T, False)
    if w_scale is not None:
        vals["w"] = (vals["w"] * np.float32(w_scale * np.sqrt(mean_deg))).astype(np.float32)
    out = dict(name=f"small{seed}", N=N, E=E, n_in=n_in, B=B, T=T, M=M,
               src=src, dst=dst, input_nodes=input_nodes)
    out.update(vals)
    out["dout"] = rs["dout"].normal(0.0, 1.0, (T, B, N)).astype(np.float32)
    return out
