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


def test_adam_update_matches_oracle():
    """Five Adam steps of the kernel, the step count advanced on the device,
    against the oracle's fp64 Adam from the same fp32 inputs."""
    import numpy as np
    import oracle
    from sparse_graph_recurrent_gb300 import _ck
    rng = np.random.default_rng(11)
    lr, b1, b2, eps = 0.01, 0.9, 0.999, 1e-8
    for n in (1, 7, 1000, 4097):
        p0 = rng.normal(size=n).astype(np.float32)
        p, m, v = torch.tensor(p0, device="cuda"), torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
        step = torch.zeros(1, dtype=torch.int64, device="cuda")
        rp, rm, rv = p0.astype(np.float64), np.zeros(n), np.zeros(n)
        for t in range(1, 6):
            g = rng.normal(size=n).astype(np.float32)
            _ck.ck_step_advance(step)
            _ck.ck_adam_update(p, torch.tensor(g, device="cuda"), m, v, step, lr, b1, b2, eps)
            rp, rm, rv = oracle.adam_update(rp, g, rm, rv, t, lr, b1, b2, eps)
        torch.cuda.synchronize()
        assert int(step.item()) == 5
        assert np.abs(p.cpu().numpy() - rp).max() <= 2e-6
        assert np.abs(m.cpu().numpy() - rm).max() <= 1e-6
        assert np.abs(v.cpu().numpy() - rv).max() <= 1e-6


def test_captured_adam_step_equals_eager_steps():
    """TrainStep with Adam: each replay advances the device step count; three
    replays equal the same calls made eagerly, bit for bit."""
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    c = workloads.small(502, 200, 8000, 10, 24, 3, 2)
    g = make_graph(c)
    lr, betas, eps = 1e-4, (0.9, 0.999), 1e-8
    M, T, B = c["M"], c["drives"].shape[0], c["state0"].shape[0]
    fixed = {k: to_dev(c[k]) for k in ("drives", "state0", "dout")}
    eager = {k: to_dev(c[k]) for k in ("w", "leak", "bias")}
    cap = {k: to_dev(c[k]) for k in ("w", "leak", "bias")}
    step = pkg.TrainStep(g, cap["w"], cap["leak"], cap["bias"], fixed["drives"], fixed["state0"],
                         fixed["dout"], M, lr, optimizer="adam", betas=betas, eps=eps)
    for k in cap:
        assert torch.equal(cap[k], eager[k])
    moments = {k: (torch.zeros_like(eager[k]), torch.zeros_like(eager[k])) for k in eager}
    count = torch.zeros(1, dtype=torch.int64, device="cuda")
    for _ in range(3):
        out_c = step().clone()
        out_e, saved, scratch = pkg.forward(g, eager["w"], eager["leak"], eager["bias"],
                                            fixed["drives"], fixed["state0"], M)
        dw, dl, db, _, _ = pkg.backward(g, eager["w"], eager["leak"], B, T, M, saved,
                                        fixed["dout"], scratch)
        _ck.ck_step_advance(count)
        for k, gr in (("w", dw), ("leak", dl), ("bias", db)):
            _ck.ck_adam_update(eager[k], gr, *moments[k], count, lr, *betas, eps)
        torch.cuda.synchronize()
        assert torch.equal(out_c, out_e)
    assert int(step.step_count.item()) == 3
    for k in cap:
        assert torch.equal(cap[k], eager[k]), k
    assert not torch.equal(cap["w"], to_dev(c["w"]))
