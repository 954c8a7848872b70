"""Graph indices in pinned host memory (CK_GRAPH_EDGES_IN_HOST_MEMORY): the
kernels read col, perm and each edge's row in place over the CPU-GPU link and
must give bitwise the results of the device-resident graph, in every launch
mode and in the recomputing variant."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import GRAD_KEYS, assert_parity, make_graph, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _default_options():
    from sparse_graph_recurrent_gb300 import _ck
    yield
    _ck.ck_set_option(_ck.OPT_PERSISTENT, 1)
    _ck.ck_set_option(_ck.OPT_GRAPH_IN_SMEM, 1)


def host_graph(c):
    import sparse_graph_recurrent_gb300 as pkg
    return pkg.SparseGraph(to_dev(c["src"]), to_dev(c["dst"]), c["N"], to_dev(c["input_nodes"]),
                           edges_in_host_memory=True)


def _assert_same(a, b):
    np.testing.assert_array_equal(a[0], b[0])
    for k in GRAD_KEYS:
        np.testing.assert_array_equal(a[1][k], b[1][k], err_msg=k)


def test_export_matches_device_graph():
    c = workloads.small(501, 300, 20000, 10, 8, 1, 1, hub_deg=9000)
    gd, gh = make_graph(c), host_graph(c)
    ed, eh = gd.export(), gh.export()
    for k in ed:
        assert torch.equal(ed[k], eh[k]), k


@pytest.mark.parametrize("seed,N,E,n_in,B,T,M,extra", [
    (502, 1, 0, 1, 1, 1, 1, {}),
    (503, 100, 3000, 8, 33, 2, 2, dict(dup_frac=0.1)),
    (504, 400, 30000, 12, 20, 3, 2, dict(hub_deg=10000)),
    (505, 120, 5000, 9, 256, 2, 2, {}),
])
def test_bitwise_equal_to_device_graph_in_every_mode(seed, N, E, n_in, B, T, M, extra):
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(seed, N, E, n_in, B, T, M, **extra)
    gd, gh = make_graph(c), host_graph(c)
    base = run_gpu(c, graph=gd)
    _assert_same(run_gpu(c, graph=gh), base)
    for opt in (_ck.OPT_GRAPH_IN_SMEM, _ck.OPT_PERSISTENT):
        _ck.ck_set_option(opt, 0)
        _assert_same(run_gpu(c, graph=gh), base)
        _ck.ck_set_option(opt, 1)
    ref_out, ref = oracle.run_case(c)
    assert_parity(*base, ref_out, ref, f"seed {seed}")


def test_flygpt_streamed_from_host_memory():
    """The FlyGPT-shaped graph with every CTA streaming its edges from host
    memory each microstep (shared-memory slices off)."""
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.make(1)
    base = run_gpu(c, graph=make_graph(c))
    gh = host_graph(c)
    _assert_same(run_gpu(c, graph=gh), base)
    _ck.ck_set_option(_ck.OPT_GRAPH_IN_SMEM, 0)
    _assert_same(run_gpu(c, graph=gh), base)


def test_recompute_with_host_graph():
    import sparse_graph_recurrent_gb300 as pkg
    c = workloads.small(506, 300, 20000, 10, 20, 2, 2, hub_deg=12000)
    base = run_gpu(c, graph=make_graph(c))
    g = host_graph(c)
    t = {k: to_dev(c[k]) for k in ("w", "leak", "bias", "drives", "state0", "dout")}
    B, T, M = c["state0"].shape[0], c["drives"].shape[0], c["M"]
    out, ckpt, scratch = pkg.forward_checkpointed(g, t["w"], t["leak"], t["bias"], t["drives"],
                                                  t["state0"], M)
    grads = pkg.backward_recompute(g, t["w"], t["leak"], t["bias"], t["drives"], B, T, M, ckpt,
                                   t["dout"], scratch)
    torch.cuda.synchronize()
    got = (out.cpu().numpy().astype(np.float64),
           {k: v.cpu().numpy().astype(np.float64) for k, v in zip(GRAD_KEYS, grads)})
    _assert_same(got, base)
