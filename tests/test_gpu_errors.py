"""Error paths of the ABI on a GPU, and the bounded device-side waits."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import assert_parity, make_graph, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def _io(c, dev="cuda"):
    return {k: to_dev(c[k]) for k in ("w", "leak", "bias", "drives", "state0", "dout")}


def test_workspace_and_shape_errors():
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(401, 50, 400, 4, 6, 2, 2)
    g = make_graph(c)
    t = _io(c)
    B, T, M = 6, 2, 2
    saved_b, scratch_b = g.workspace_size(B, T, M)
    out = torch.empty((T, B, 50), device="cuda")
    saved = torch.empty(saved_b, dtype=torch.uint8, device="cuda")
    scratch = torch.empty(scratch_b, dtype=torch.uint8, device="cuda")
    small = torch.empty(saved_b - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_ck.CKError) as e:
        _ck.ck_forward(g.handle, t["w"], t["leak"], t["bias"], t["drives"], t["state0"], M, out,
                       small, scratch)
    assert e.value.name == "CK_ERR_WORKSPACE"
    for bad in ((0, 1, 1), (1, 0, 1), (1, 1, 0)):
        with pytest.raises(_ck.CKError) as e:
            g.workspace_size(*bad)
        assert e.value.name == "CK_ERR_INVALID_ARG"
    with pytest.raises(_ck.CKError) as e:
        g.workspace_size(513, 1, 1)
    assert e.value.name == "CK_ERR_UNSUPPORTED"
    lib = _ck.load()
    st = lib.ck_forward(g.handle, None, None, None, None, None, B, T, M, None, None, 0, None, 0, None)
    assert st == 1
    # the graph still works after the refusals
    out2, grads = run_gpu(c, graph=g)
    ref_out, ref = oracle.run_case(c)
    assert_parity(out2, grads, ref_out, ref, "after errors")


@pytest.mark.parametrize("streamed", [False, True], ids=["graph_in_smem", "graph_streamed"])
def test_barrier_timeout_is_reported_and_context_survives(streamed):
    """Barriers are told to wait for one more CTA than exists; every wait runs
    out after 2 ms, the kernel stops, and the status word says so -- in the
    forward and in the backward, with the graph slice in shared memory and
    streamed (where the ring's copies are in flight when the wait gives up)."""
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(402, 60, 600, 4, 8, 2, 2)
    g = make_graph(c)
    t = _io(c)
    B, T, M = c["B"], c["T"], c["M"]
    _ck.ck_set_option(_ck.OPT_GRAPH_IN_SMEM, 0 if streamed else 1)
    _ck.ck_set_option(_ck.OPT_BARRIER_TIMEOUT_NS, 2_000_000)
    try:
        _ck.ck_set_option(_ck.OPT_TEST_BARRIER_EXTRA, 1)
        out, saved, scratch = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"],
                                          t["state0"], M)
        with pytest.raises(_ck.CKError) as e:
            _ck.ck_query_status(scratch)
        assert e.value.name == "CK_ERR_TIMEOUT"
        # a complete forward, then a backward whose barriers run out
        _ck.ck_set_option(_ck.OPT_TEST_BARRIER_EXTRA, 0)
        out, saved, scratch = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"],
                                          t["state0"], M)
        _ck.ck_query_status(scratch)
        _ck.ck_set_option(_ck.OPT_TEST_BARRIER_EXTRA, 1)
        pkg.backward(g, t["w"], t["leak"], B, T, M, saved, t["dout"], scratch)
        with pytest.raises(_ck.CKError) as e:
            _ck.ck_query_status(scratch)
        assert e.value.name == "CK_ERR_TIMEOUT"
    finally:
        _ck.ck_set_option(_ck.OPT_TEST_BARRIER_EXTRA, 0)
        _ck.ck_set_option(_ck.OPT_BARRIER_TIMEOUT_NS, 4_000_000_000)
    try:
        out, grads = run_gpu(c, graph=g)
    finally:
        _ck.ck_set_option(_ck.OPT_GRAPH_IN_SMEM, 1)
    ref_out, ref = oracle.run_case(c)
    assert_parity(out, grads, ref_out, ref, "after timeout")


def test_binding_rejects_wrong_shapes_before_any_launch():
    """The library sees only pointers; the binding checks every shape against
    the graph and the call, so a mismatched tensor never reaches a kernel."""
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(402, 40, 300, 4, 5, 2, 2)
    g = make_graph(c)
    t = _io(c)
    B, T, M = 5, 2, 2
    saved_b, scratch_b = g.workspace_size(B, T, M)
    out = torch.empty((T, B, 40), device="cuda")
    saved = torch.empty(saved_b, dtype=torch.uint8, device="cuda")
    scratch = torch.empty(scratch_b, dtype=torch.uint8, device="cuda")
    bad = {
        "drives": t["drives"][:, :3].contiguous(),        # n_in 3 instead of 4
        "leak": t["leak"][:39].contiguous(),               # N - 1
        "w": t["w"][:-1].contiguous(),                      # E - 1
    }
    for name, tensor in bad.items():
        args = dict(t, **{name: tensor})
        with pytest.raises(ValueError):
            _ck.ck_forward(g.handle, args["w"], args["leak"], args["bias"], args["drives"],
                           args["state0"], M, out, saved, scratch)
    with pytest.raises(ValueError):
        _ck.ck_forward(g.handle, t["w"], t["leak"], t["bias"], t["drives"], t["state0"], M,
                       torch.empty((T, B, 41), device="cuda"), saved, scratch)
