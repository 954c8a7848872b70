"""A whole training step (forward, backward, SGD update of edge values, leak
and bias) captured as one CUDA graph: replays equal the same calls made
eagerly, bit for bit."""
import pytest
import torch

import workloads
from gpu_helpers import make_graph, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cid_or_small", ["small", 1])
def test_captured_step_equals_eager_steps(cid_or_small):
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(501, 200, 8000, 10, 24, 3, 2) if cid_or_small == "small" else workloads.make(1)
    g = make_graph(c)
    # small enough that leak stays in (0, 1) over the steps (it is updated unsquashed)
    lr = 1e-3 if cid_or_small == "small" else 1e-7
    M, T, B = c["M"], c["drives"].shape[0], c["state0"].shape[0]
    fixed = {k: to_dev(c[k]) for k in ("drives", "state0", "dout")}
    eager = {k: to_dev(c[k]) for k in ("w", "leak", "bias")}
    cap = {k: to_dev(c[k]) for k in ("w", "leak", "bias")}
    step = pkg.TrainStep(g, cap["w"], cap["leak"], cap["bias"], fixed["drives"], fixed["state0"],
                         fixed["dout"], M, lr)
    # the setup pass leaves the parameters untouched
    for k in cap:
        assert torch.equal(cap[k], eager[k])
    for _ in range(3):
        out_c = step().clone()
        out_e, saved, scratch = pkg.forward(g, eager["w"], eager["leak"], eager["bias"],
                                            fixed["drives"], fixed["state0"], M)
        dw, dl, db, _, _ = pkg.backward(g, eager["w"], eager["leak"], B, T, M, saved,
                                        fixed["dout"], scratch)
        _ck.ck_sgd_update(eager["w"], dw, lr)
        _ck.ck_sgd_update(eager["leak"], dl, lr)
        _ck.ck_sgd_update(eager["bias"], db, lr)
        torch.cuda.synchronize()
        assert torch.isfinite(out_c).all()
        assert torch.equal(out_c, out_e)
    for k in cap:
        assert torch.equal(cap[k], eager[k]), k
    assert not torch.equal(cap["w"], to_dev(c["w"]))  # the step did move the parameters


def test_sgd_update_matches_torch():
    from sparse_graph_recurrent_gb300 import _ck
    for n in (0, 1, 7, 1000, 4097):
        p = torch.randn(n, device="cuda")
        g = torch.randn(n, device="cuda")
        ref = p - 0.01 * g
        _ck.ck_sgd_update(p, g, 0.01)
        torch.cuda.synchronize()
        assert torch.allclose(p, ref, rtol=0, atol=1e-6)
