"""ck_forward_static_scratch: the forward for callers that cannot allocate
device memory (a plugin whose host application's memory manager owns the
device, a control loop that must not allocate once running).  Its workspace is
an array compiled into the library, so the test checks it against ck_forward
with a caller-allocated scratch buffer, on two calls in a row with different
inputs: the shared array must not carry anything from one call into the next.

This file is collected last on purpose; it must pass on its own in a fresh
process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_helpers import STATE_TOL, make_graph, to_dev

pytestmark = pytest.mark.gpu


def _inputs(c, seed_shift):
    rng = np.random.default_rng(seed_shift)
    state0 = c["state0"] if seed_shift == 0 else (0.1 * rng.normal(size=c["state0"].shape)).astype(np.float32)
    drives = c["drives"] if seed_shift == 0 else rng.normal(size=c["drives"].shape).astype(np.float32)
    return {k: to_dev(v) for k, v in dict(w=c["w"], leak=c["leak"], bias=c["bias"], drives=drives,
                                        state0=state0).items()}


def test_static_scratch_forward_matches_ck_forward_twice():
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(901, 700, 40000, 12, 20, 4, 2, hub_deg=9000)
    g = make_graph(c)
    B, T, M, N = c["B"], c["T"], c["M"], c["N"]
    for call in range(2):
        t = _inputs(c, call)
        want, _, _ = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"], t["state0"], M)
        saved_b, _ = g.workspace_size(B, T, M)
        saved = torch.empty(saved_b, dtype=torch.uint8, device="cuda")
        got = torch.full((T, B, N), float("nan"), device="cuda")
        _ck.ck_forward_static_scratch(g.handle, t["w"], t["leak"], t["bias"], t["drives"],
                                      t["state0"], M, got, saved)
        torch.cuda.synchronize()
        err = (got - want).abs().max().item()
        assert err <= STATE_TOL, (call, err)


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
