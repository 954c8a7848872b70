"""The context-only torch.sparse baseline in bench.py computes the same step:
on the CPU in fp64 it matches the oracle on the tiny workload."""
import numpy as np
import torch

import bench
import oracle
import workloads
from gpu_helpers import GRAD_KEYS, rel_err


def test_torch_sparse_step_matches_oracle():
    c = workloads.make(0)
    out, grads = bench.torch_sparse_step(c, torch.device("cpu"), torch.float64)
    ref_out, ref = oracle.run_case(c)
    got = out.numpy()
    assert np.abs(got - ref_out).max() <= 1e-10
    for k, g in zip(GRAD_KEYS, grads):
        g = g.to_dense() if g.is_sparse else g
        assert rel_err(g.numpy(), ref[k]) <= 1e-10, k
