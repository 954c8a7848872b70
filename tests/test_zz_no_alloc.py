"""ck_forward_static_scratch: the forward for callers that cannot allocate
device memory (a plugin whose host application's memory manager owns the
device, a control loop that must not allocate once running).  Its workspace is
an array compiled into the library, so the tests check it against ck_forward
with a caller-allocated scratch buffer, on two calls in a row with different
inputs: the shared array must not carry anything from one call into the next.
Both entry points run the same kernels on the same inputs, so their outputs
and `saved` must agree bit for bit, and a backward from the static path's
`saved` must give ck_backward's gradients bit for bit.

This file is collected last on purpose; it must pass on its own in a fresh
process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import make_graph, to_dev

pytestmark = pytest.mark.gpu


def _inputs(c, seed_shift):
    rng = np.random.default_rng(seed_shift)
    state0 = c["state0"] if seed_shift == 0 else (0.1 * rng.normal(size=c["state0"].shape)).astype(np.float32)
    drives = c["drives"] if seed_shift == 0 else rng.normal(size=c["drives"].shape).astype(np.float32)
    return {k: to_dev(v) for k, v in dict(w=c["w"], leak=c["leak"], bias=c["bias"], drives=drives,
                                        state0=state0, dout=c["dout"]).items()}


@pytest.fixture
def _options():
    """Set library options for one test and restore the defaults after it."""
    from sparse_graph_recurrent_gb300 import _ck
    defaults = {_ck.OPT_PERSISTENT: 1, _ck.OPT_GRAPH_IN_SMEM: 1, _ck.OPT_ROWS_IN_SMEM: 1,
                _ck.OPT_TEST_BARRIER_EXTRA: 0, _ck.OPT_BARRIER_TIMEOUT_NS: 4_000_000_000}

    def set_(**kv):
        for name, v in kv.items():
            _ck.ck_set_option(getattr(_ck, "OPT_" + name), v)
    yield set_
    for opt, v in defaults.items():
        _ck.ck_set_option(opt, v)


# the default launch; the graph streamed and row sums in the scratch array
# (the array's permuted-value and row-sum regions); one launch per microstep
MODES = {
    "persistent": {},
    "streamed_rows_global": {"GRAPH_IN_SMEM": 0, "ROWS_IN_SMEM": 0},
    "launch_per_microstep": {"PERSISTENT": 0},
}


@pytest.mark.parametrize("mode", list(MODES))
def test_static_scratch_forward_matches_ck_forward_twice(_options, mode):
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    _options(**MODES[mode])
    c = workloads.small(901, 700, 40000, 12, 20, 4, 2, hub_deg=9000)
    g = make_graph(c)
    B, T, M, N = c["B"], c["T"], c["M"], c["N"]
    for call in range(2):
        t = _inputs(c, call)
        want, want_saved, scratch = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"],
                                                t["state0"], M)
        _ck.ck_query_status(scratch)
        saved_b, _ = g.workspace_size(B, T, M)
        saved = torch.full((saved_b,), 0xAB, dtype=torch.uint8, device="cuda")
        got = torch.full((T, B, N), float("nan"), device="cuda")
        _ck.ck_forward_static_scratch(g.handle, t["w"], t["leak"], t["bias"], t["drives"],
                                      t["state0"], M, got, saved)
        _ck.ck_query_status_static()
        assert torch.equal(got, want), (mode, call, (got - want).abs().max().item())
        assert torch.equal(saved, want_saved), (mode, call)
        # the static path's saved activations feed the ordinary backward
        g_static = pkg.backward(g, t["w"], t["leak"], B, T, M, saved, t["dout"], scratch)
        g_want = pkg.backward(g, t["w"], t["leak"], B, T, M, want_saved, t["dout"], scratch)
        _ck.ck_query_status(scratch)
        for a, b in zip(g_static, g_want):
            assert torch.equal(a, b), (mode, call)


def test_static_scratch_reports_a_wait_that_ran_out(_options):
    """A bounded device-side wait that gives up is reported by
    ck_query_status_static (the status word lives in the static array), and the
    next call is correct again."""
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(903, 60, 600, 4, 8, 2, 2)
    g = make_graph(c)
    B, T, M, N = c["B"], c["T"], c["M"], c["N"]
    t = _inputs(c, 0)
    saved_b, _ = g.workspace_size(B, T, M)
    saved = torch.empty(saved_b, dtype=torch.uint8, device="cuda")
    got = torch.empty((T, B, N), device="cuda")
    _options(BARRIER_TIMEOUT_NS=2_000_000, TEST_BARRIER_EXTRA=1)
    _ck.ck_forward_static_scratch(g.handle, t["w"], t["leak"], t["bias"], t["drives"],
                                  t["state0"], M, got, saved)
    with pytest.raises(_ck.CKError) as e:
        _ck.ck_query_status_static()
    assert e.value.name == "CK_ERR_TIMEOUT"
    _options(BARRIER_TIMEOUT_NS=4_000_000_000, TEST_BARRIER_EXTRA=0)
    _ck.ck_forward_static_scratch(g.handle, t["w"], t["leak"], t["bias"], t["drives"],
                                  t["state0"], M, got, saved)
    _ck.ck_query_status_static()
    want, _, scratch = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"], t["state0"], M)
    _ck.ck_query_status(scratch)
    assert torch.equal(got, want)


def test_static_scratch_rejects_shapes_beyond_the_array():
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(902, 3000, 9_000_000, 4, 32, 1, 1)
    g = make_graph(c)
    N, B, T, M = c["N"], c["B"], c["T"], c["M"]
    t = _inputs(c, 0)
    saved_b, _ = g.workspace_size(B, T, M)
    saved = torch.empty(saved_b, dtype=torch.uint8, device="cuda")
    out = torch.empty((T, B, N), device="cuda")
    with pytest.raises(_ck.CKError) as e:
        _ck.ck_forward_static_scratch(g.handle, t["w"], t["leak"], t["bias"], t["drives"],
                                      t["state0"], M, out, saved)
    assert e.value.name == "CK_ERR_UNSUPPORTED" and "static array" in str(e.value)
