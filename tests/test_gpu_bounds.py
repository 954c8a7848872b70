"""The bounds-checked build of the library (compiled with -DCK_DEBUG_BOUNDS).

In that build every gathered row, table and carry index the kernels compute
from graph data is checked on the device; a bad one is recorded in the status
word (ck_query_status then reports CK_ERR_INTERNAL) and its access is skipped.
The tests run the small parity cases and the tiny workload against the oracle
in a child process that loads that build, expecting every call to report
CK_OK, and check with the probe hook that a bad index is reported.

Each test starts its own Python process because a process loads one variant
of the library (CK_LIBRARY_VARIANT=bounds selects libck_bounds.so).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _child_env():
    env = dict(os.environ)
    env["CK_LIBRARY_VARIANT"] = "bounds"
    return env


def test_bounds_build_small_cases_report_ok():
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_parity.py"),
                        "-k", "small_cases or config0 or modes_are_bitwise"],
                       cwd=ROOT, env=_child_env(), capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


CHILD = r'''
import sys
sys.path.insert(0, "tests")
import torch
import workloads
import sparse_graph_recurrent_gb300 as pkg
from sparse_graph_recurrent_gb300 import _ck
from gpu_helpers import make_graph, to_dev
assert _ck.library_path().endswith("libck_bounds.so"), _ck.library_path()
c = workloads.small(905, 90, 900, 4, 8, 2, 2)
g = make_graph(c)
t = {k: to_dev(c[k]) for k in ("w", "leak", "bias", "drives", "state0")}
_ck.ck_set_option(_ck.OPT_TEST_BOUNDS_PROBE, 1)
out, saved, scratch = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"], t["state0"], c["M"])
try:
    _ck.ck_query_status(scratch)
    raise SystemExit("the probe index was not reported")
except _ck.CKError as e:
    assert e.name == "CK_ERR_INTERNAL" and "out of bounds" in str(e), str(e)
_ck.ck_set_option(_ck.OPT_TEST_BOUNDS_PROBE, 0)
out2, saved2, scratch2 = pkg.forward(g, t["w"], t["leak"], t["bias"], t["drives"], t["state0"], c["M"])
_ck.ck_query_status(scratch2)
# a recorded error stops the flagged kernel at its next barrier (its outputs are
# partial); the next call, with the hook off, is complete and matches the oracle
import numpy as np
import oracle
ref_out, _ = oracle.run_case(c)
assert np.abs(out2.cpu().numpy() - ref_out).max() <= 1e-5
print("probe ok")
'''


def test_bounds_build_reports_a_bad_index():
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=_child_env(),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "probe ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
