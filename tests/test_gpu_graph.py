"""GPU graph build (ck_graph_create) against hand-derived layouts and the
oracle's stable sort: bit-exact on every array."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from golden_io import read_cases
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

KEYS = ("row_ptr", "col", "perm", "rowT_ptr", "colT", "permT", "slot")


def _export(N, src, dst, inp):
    import sparse_graph_recurrent_gb300 as pkg
    g = pkg.SparseGraph(to_dev(np.asarray(src, np.int64)), to_dev(np.asarray(dst, np.int64)), N,
                        to_dev(np.asarray(inp, np.int64)))
    out = {k: v.cpu().numpy().astype(np.int64) for k, v in g.export().items()}
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("case", read_cases("csr_tiny.txt"), ids=lambda c: c["name"])
def test_hand_derived_layouts(case):
    got = _export(case["N"], case["src"], case["dst"], case["input_nodes"])
    for k in KEYS:
        np.testing.assert_array_equal(got[k], case[k], err_msg=k)


@pytest.mark.parametrize("seed,N,E,hub", [(1, 1, 0, 0), (2, 1, 7, 0), (3, 9, 0, 0), (4, 300, 5000, 0),
                                          (5, 70000, 100000, 40000), (6, 3, 20000, 0)])
def test_random_graphs_match_oracle(seed, N, E, hub):
    c = workloads.small(seed, N, E, min(5, N), 1, 1, 1, dup_frac=0.1, hub_deg=hub)
    got = _export(N, c["src"], c["dst"], c["input_nodes"])
    want = oracle.graph_layout(N, c["src"], c["dst"], c["input_nodes"])
    for k in KEYS:
        np.testing.assert_array_equal(got[k], want[k].astype(np.int64), err_msg=k)


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4])
def test_workload_graphs_match_oracle(cid):
    c = workloads.make(cid, with_dout=False)
    got = _export(c["N"], c["src"], c["dst"], c["input_nodes"])
    want = oracle.graph_layout(c["N"], c["src"], c["dst"], c["input_nodes"])
    for k in KEYS:
        np.testing.assert_array_equal(got[k], want[k].astype(np.int64), err_msg=k)


def test_bad_graphs_are_rejected():
    from sparse_graph_recurrent_gb300 import _ck
    bad = [([0, 5], [1, 1], [0], "edge endpoint"),      # src out of range
           ([0, 1], [1, -1], [0], "edge endpoint"),     # dst negative
           ([0, 1], [1, 2], [0, 3], "input node"),      # input out of range
           ([0, 1], [1, 2], [2, 0, 2], "repeats")]      # duplicate input
    for src, dst, inp, msg in bad:
        with pytest.raises(_ck.CKError) as e:
            _export(3, src, dst, inp)
        assert e.value.name == "CK_ERR_INVALID_ARG" and msg in str(e.value)
    # the context is still usable afterwards
    got = _export(3, [0, 1], [1, 2], [0])
    np.testing.assert_array_equal(got["row_ptr"], [0, 0, 1, 2])
