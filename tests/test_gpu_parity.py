"""CUDA path (through the C ABI) against the oracle on identical seeded inputs.

Tolerances: states within 1e-5 max-abs; each of the five gradients within
1e-4 of max-abs error over the oracle's max-abs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import (GRAD_KEYS, assert_parity, make_graph, rel_err, run_gpu, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _default_options():
    from sparse_graph_recurrent_gb300 import _ck
    yield
    _ck.ck_set_option(_ck.OPT_PERSISTENT, 1)
    _ck.ck_set_option(_ck.OPT_GRAPH_IN_SMEM, 1)
    _ck.ck_set_option(_ck.OPT_ROWS_IN_SMEM, 1)
    _ck.ck_set_option(_ck.OPT_TILED, 0)


# The two kernel families: the tiled kernels (state chunks gathered from shared
# memory; used when the graph has a tiling and B <= 32) and the L2-gather
# kernels (every other shape, and all shapes with the tiled kernels off).
KERNELS = {"tiled": 1, "l2": 0}


def _kernels(name):
    from sparse_graph_recurrent_gb300 import _ck
    _ck.ck_set_option(_ck.OPT_TILED, KERNELS[name])


SMALL = [
    # seed, N, E, n_in, B, T, M, extra
    (101, 1, 0, 1, 1, 1, 1, {}),
    (102, 2, 3, 1, 3, 2, 2, {}),
    (103, 17, 60, 4, 8, 3, 1, dict(dup_frac=0.2)),
    (104, 40, 0, 5, 5, 2, 3, {}),
    (105, 64, 900, 6, 20, 2, 2, dict(hub_deg=400)),
    (106, 100, 3000, 8, 31, 2, 3, dict(dup_frac=0.1)),
    (107, 100, 3000, 8, 32, 3, 2, {}),
    (108, 100, 3000, 8, 33, 2, 1, {}),
    (109, 300, 20000, 10, 64, 1, 2, dict(hub_deg=12000)),
    (110, 200, 8000, 10, 129, 2, 2, {}),
    (111, 150, 6000, 7, 200, 1, 3, dict(hub_deg=3000)),
    (112, 120, 5000, 9, 256, 2, 2, {}),
    (113, 90, 4000, 9, 300, 1, 2, {}),
    (114, 60, 2500, 4, 512, 1, 1, {}),
    (115, 3000, 200000, 32, 32, 2, 2, dict(hub_deg=150000)),
    # one source feeding 4,000 edges: a hub row of the backward's transposed rows
    (116, 500, 6000, 8, 16, 2, 2, dict(src_hub_deg=4000)),
    # mostly empty rows (E << N): pieces of many rows and few edges
    (117, 30000, 5000, 16, 5, 2, 2, {}),
    # self-loops only: every node its own scalar recurrence
    (118, 300, 900, 4, 8, 3, 3, dict(loops_only=True)),
    # no input nodes: drives [T, 0, B], and d_drives empty
    (119, 50, 400, 0, 4, 2, 2, {}),
]


@pytest.mark.parametrize("kernels", list(KERNELS))
@pytest.mark.parametrize("seed,N,E,n_in,B,T,M,extra", SMALL, ids=[f"s{c[0]}_N{c[1]}_E{c[2]}_B{c[4]}_M{c[6]}" for c in SMALL])
def test_small_cases(seed, N, E, n_in, B, T, M, extra, kernels):
    _kernels(kernels)
    c = workloads.small(seed, N, E, n_in, B, T, M, **extra)
    out, g = run_gpu(c)
    ref_out, ref = oracle.run_case(c)
    assert_parity(out, g, ref_out, ref, f"seed {seed}")


def test_two_graphs_interleaved():
    """Handles are independent: two graphs alive at once, their forward and
    backward calls interleaved, each give what they give alone."""
    import sparse_graph_recurrent_gb300 as pkg
    ca = workloads.small(121, 400, 9000, 6, 16, 2, 2, hub_deg=3000)
    cb = workloads.small(122, 900, 20000, 12, 33, 3, 1, dup_frac=0.1)
    alone = {k: run_gpu(c) for k, c in (("a", ca), ("b", cb))}
    ga, gb = make_graph(ca), make_graph(cb)
    ta = {k: to_dev(ca[k]) for k in ("w", "leak", "bias", "drives", "state0", "dout")}
    tb = {k: to_dev(cb[k]) for k in ("w", "leak", "bias", "drives", "state0", "dout")}
    oa, sa, xa = pkg.forward(ga, ta["w"], ta["leak"], ta["bias"], ta["drives"], ta["state0"], ca["M"])
    ob, sb, xb = pkg.forward(gb, tb["w"], tb["leak"], tb["bias"], tb["drives"], tb["state0"], cb["M"])
    da = pkg.backward(ga, ta["w"], ta["leak"], ca["B"], ca["T"], ca["M"], sa, ta["dout"], xa)
    db = pkg.backward(gb, tb["w"], tb["leak"], cb["B"], cb["T"], cb["M"], sb, tb["dout"], xb)
    torch.cuda.synchronize()
    for (out, grads), (o, d) in ((alone["a"], (oa, da)), (alone["b"], (ob, db))):
        np.testing.assert_array_equal(o.cpu().numpy().astype(np.float64), out)
        for k, v in zip(GRAD_KEYS, d):
            np.testing.assert_array_equal(v.cpu().numpy().astype(np.float64), grads[k], err_msg=k)


def test_side_stream_gives_the_same_bits():
    """Every call enqueues on the caller's stream: the same case built and run
    inside a side stream (graph build, workspaces, launches and copies) gives
    the default stream's outputs and gradients bit for bit."""
    c = workloads.small(120, 700, 30000, 10, 32, 3, 2, hub_deg=9000)
    base_out, base = run_gpu(c)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        out, g = run_gpu(c)
    side.synchronize()
    np.testing.assert_array_equal(out, base_out)
    for k in GRAD_KEYS:
        np.testing.assert_array_equal(g[k], base[k], err_msg=k)


@pytest.mark.parametrize("kernels", list(KERNELS))
def test_config0_tiny(kernels):
    _kernels(kernels)
    c = workloads.make(0)
    out, g = run_gpu(c)
    ref_out, ref = oracle.run_case(c)
    assert_parity(out, g, ref_out, ref, "tiny")


_ORACLE = {}


def _oracle_full(cid, M=None):
    """The oracle's full run of a workload, computed once per test session."""
    key = (cid, M)
    if key not in _ORACLE:
        c = workloads.make(cid, M=M)
        _ORACLE[key] = (c, oracle.step_columns(c, oracle.threads_available()))
    return _ORACLE[key]


@pytest.mark.slow
@pytest.mark.parametrize("kernels", list(KERNELS))
def test_config1_flygpt_full(kernels):
    _kernels(kernels)
    c, (ref_out, ref) = _oracle_full(1)
    out, g = run_gpu(c)
    assert_parity(out, g, ref_out, ref, "flygpt")


@pytest.mark.slow
@pytest.mark.parametrize("kernels", list(KERNELS))
@pytest.mark.parametrize("M", [1, 2, 3])
def test_config2_ragged_full(M, kernels):
    _kernels(kernels)
    c, (ref_out, ref) = _oracle_full(2, M)
    out, g = run_gpu(c)
    assert_parity(out, g, ref_out, ref, f"ragged M={M}")


def _sampled(cid, cols):
    """Full-size run on the GPU; the loss only weighs the sampled batch columns,
    so every gradient equals the oracle's on those columns alone."""
    c = workloads.make(cid)
    mask = np.zeros_like(c["dout"])
    mask[:, cols, :] = c["dout"][:, cols, :]
    out, g = run_gpu(c, dout=mask)
    c["dout"] = mask
    ref_out, ref = oracle.run_case(c, batch_cols=cols)
    e = np.abs(out[:, cols, :] - ref_out).max()
    assert e <= 1e-5, e
    got = dict(g)
    got["ddrives"] = g["ddrives"][:, :, cols]
    got["dstate0"] = g["dstate0"][cols]
    for k in GRAD_KEYS:
        assert rel_err(got[k], ref[k]) <= 1e-4, (k, rel_err(got[k], ref[k]))
    # columns outside the sample carry no gradient at all
    rest = np.setdiff1d(np.arange(c["state0"].shape[0]), cols)
    assert np.all(g["dstate0"][rest] == 0) and np.all(g["ddrives"][:, :, rest] == 0)


@pytest.mark.slow
def test_config3_wide_sampled_columns():
    _sampled(3, [0, 131])


@pytest.mark.slow
def test_config4_connectome_sampled_column():
    _sampled(4, [19])


@pytest.mark.parametrize("kernels", list(KERNELS))
def test_modes_are_bitwise_identical(kernels):
    """One launch per microstep (operands read from global memory), the graph
    streamed from global memory, and row sums kept in the scratch buffer follow
    the same summation order as the default persistent launch."""
    from sparse_graph_recurrent_gb300 import _ck
    _kernels(kernels)
    c = workloads.small(201, 400, 30000, 12, 20, 3, 2, hub_deg=10000)
    base_out, base = run_gpu(c)
    again_out, again = run_gpu(c)
    np.testing.assert_array_equal(base_out, again_out)
    for opt, val in ((_ck.OPT_PERSISTENT, 0), (_ck.OPT_GRAPH_IN_SMEM, 0), (_ck.OPT_ROWS_IN_SMEM, 0)):
        _ck.ck_set_option(opt, val)
        out, g = run_gpu(c)
        _ck.ck_set_option(opt, 1)
        np.testing.assert_array_equal(out, base_out)
        for k in GRAD_KEYS:
            np.testing.assert_array_equal(g[k], base[k])
    ref_out, ref = oracle.run_case(c)
    assert_parity(base_out, base, ref_out, ref, "persistent")


def test_autograd_function_matches_oracle():
    import sparse_graph_recurrent_gb300 as pkg
    c = workloads.small(301, 80, 2000, 6, 12, 3, 2)
    g = make_graph(c)
    leaves = {k: to_dev(c[k]).requires_grad_() for k in ("w", "leak", "bias", "drives", "state0")}
    out = pkg.sparse_recurrence(leaves["w"], leaves["leak"], leaves["bias"], leaves["drives"],
                                leaves["state0"], g, microsteps=c["M"])
    (out * to_dev(c["dout"])).sum().backward()
    ref_out, ref = oracle.run_case(c)
    grads = {k2: leaves[k1].grad.cpu().numpy().astype(np.float64)
             for k1, k2 in zip(("w", "leak", "bias", "drives", "state0"), GRAD_KEYS)}
    assert_parity(out.detach().cpu().numpy().astype(np.float64), grads, ref_out, ref, "autograd")
