"""The recomputing variant (ck_forward_checkpointed + ck_backward_recompute)
against the regular calls, bit for bit, and against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import GRAD_KEYS, assert_parity, make_graph, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # seed, N, E, n_in, B, T, M, extra
    (401, 1, 0, 1, 1, 1, 1, {}),
    (402, 40, 300, 4, 8, 1, 3, {}),
    (403, 100, 3000, 8, 32, 3, 2, dict(dup_frac=0.1)),
    (404, 300, 20000, 10, 20, 2, 1, dict(hub_deg=12000)),
    (405, 200, 8000, 10, 64, 2, 3, {}),
    (406, 90, 4000, 9, 300, 2, 2, {}),
    (407, 60, 900, 0, 8, 3, 2, {}),  # no input nodes: drives and their gradient are empty
]


def _both(c):
    import sparse_graph_recurrent_gb300 as pkg
    g = make_graph(c)
    t = {k: to_dev(c[k]) for k in ("w", "leak", "bias", "drives", "state0", "dout")}
    B, T, M = c["state0"].shape[0], c["drives"].shape[0], c["M"]
    out, saved, _ = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"], t["state0"], M)
    grads = pkg.backward(g, t["w"], t["leak"], B, T, M, saved, t["dout"])
    rout, ckpt, scratch = pkg.forward_checkpointed(g, t["w"], t["leak"], t["bias"], t["drives"],
                                                   t["state0"], M)
    rgrads = pkg.backward_recompute(g, t["w"], t["leak"], t["bias"], t["drives"], B, T, M, ckpt,
                                    t["dout"], scratch)
    torch.cuda.synchronize()
    return (g, out, saved, grads), (rout, ckpt, rgrads)


def _check_identical(c):
    (g, out, saved, grads), (rout, ckpt, rgrads) = _both(c)
    assert torch.equal(out, rout)
    # checkpoint t is the saved state entering input step t (node-major rows)
    N, T, M = c["N"], c["drives"].shape[0], c["M"]
    H = saved.view(torch.float32)
    C = ckpt.view(torch.float32)
    Bp = C.numel() // ((T + 1) * N)
    for t in range(T + 1):
        assert torch.equal(C[t * N * Bp:(t + 1) * N * Bp], H[t * M * N * Bp:(t * M + 1) * N * Bp])
    for k, a, b in zip(GRAD_KEYS, grads, rgrads):
        assert torch.equal(a, b), k


@pytest.mark.parametrize("seed,N,E,n_in,B,T,M,extra", CASES,
                         ids=[f"r{c[0]}_B{c[4]}_T{c[5]}_M{c[6]}" for c in CASES])
def test_recompute_is_bitwise_identical(seed, N, E, n_in, B, T, M, extra):
    _check_identical(workloads.small(seed, N, E, n_in, B, T, M, **extra))


def test_recompute_flygpt_bitwise_identical():
    _check_identical(workloads.make(1))


@pytest.fixture
def _recompute_steps():
    from sparse_graph_recurrent_gb300 import _ck
    yield lambda k: _ck.ck_set_option(_ck.OPT_RECOMPUTE_STEPS, k)
    _ck.ck_set_option(_ck.OPT_RECOMPUTE_STEPS, 0)


@pytest.mark.parametrize("K", [1, 2, 3, 5, 7, 9])
@pytest.mark.parametrize("M", [1, 3])
def test_windows_of_several_steps_are_bitwise_identical(_recompute_steps, K, M):
    """Windows of K input steps, including a shorter lowest window (T = 7)
    and K beyond T (clamped to one window)."""
    _recompute_steps(K)
    _check_identical(workloads.small(409 + M, 200, 8000, 10, 20, 7, M, hub_deg=3000))


def test_window_size_sets_the_scratch(_recompute_steps):
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(412, 300, 5000, 6, 32, 16, 2)
    g = make_graph(c)
    N, Bp = c["N"], 32
    sizes = {}
    for K in (1, 4, 16, 0):
        _recompute_steps(K)
        sizes[K] = _ck.ck_workspace_size_recompute(g.handle, 32, 16, 2)[1]
    assert sizes[0] == sizes[4]  # round(sqrt(16))
    # each extra input step in the window holds M more states and M more proposals
    assert sizes[16] - sizes[4] == 12 * 2 * 2 * N * Bp * 4
    assert sizes[4] - sizes[1] == 3 * 2 * 2 * N * Bp * 4


def test_recompute_autograd_matches_oracle():
    import sparse_graph_recurrent_gb300 as pkg
    c = workloads.small(407, 150, 6000, 7, 24, 3, 2, hub_deg=2000)
    g = make_graph(c)
    leaves = {k: to_dev(c[k]).requires_grad_() for k in ("w", "leak", "bias", "drives", "state0")}
    out = pkg.sparse_recurrence(leaves["w"], leaves["leak"], leaves["bias"], leaves["drives"],
                                leaves["state0"], g, microsteps=c["M"], recompute=True)
    (out * to_dev(c["dout"])).sum().backward()
    ref_out, ref = oracle.run_case(c)
    grads = {k2: leaves[k1].grad.cpu().numpy().astype(np.float64)
             for k1, k2 in zip(("w", "leak", "bias", "drives", "state0"), GRAD_KEYS)}
    assert_parity(out.detach().cpu().numpy().astype(np.float64), grads, ref_out, ref, "recompute")


def test_recompute_workspace_is_checked():
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(408, 50, 500, 5, 8, 2, 2)
    g = make_graph(c)
    t = {k: to_dev(c[k]) for k in ("w", "leak", "bias", "drives", "state0")}
    ckpt_b, scratch_b = _ck.ck_workspace_size_recompute(g.handle, 8, 2, 2)
    out = torch.empty((2, 8, 50), device="cuda")
    ckpt = torch.empty(ckpt_b - 16, dtype=torch.uint8, device="cuda")
    scratch = torch.empty(scratch_b, dtype=torch.uint8, device="cuda")
    with pytest.raises(_ck.CKError) as ei:
        _ck.ck_forward_checkpointed(g.handle, t["w"], t["leak"], t["bias"], t["drives"],
                                    t["state0"], 2, out, ckpt, scratch)
    assert ei.value.name == "CK_ERR_WORKSPACE"
