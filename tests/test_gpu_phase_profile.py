"""The profiling build (libck_prof.so, -DCK_PHASE_PROFILE): its phase counters
add up per CTA, and its results still match the oracle; and every build of the
library (ordinary, bounds-checked, profiling) gives the same bits.

A process loads one variant of the library, so the checks run in a child
process with CK_LIBRARY_VARIANT=prof.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, "tests")
import numpy as np
import oracle
import workloads
from sparse_graph_recurrent_gb300 import _ck
from gpu_helpers import assert_parity, run_gpu
assert _ck.library_path().endswith("libck_prof.so"), _ck.library_path()
c = workloads.small(921, 400, 12000, 8, 16, 3, 2, hub_deg=3000)
S = c["drives"].shape[0] * c["M"]
_ck.ck_phase_profile_read(clear=True)
out, grads = run_gpu(c)
data = _ck.ck_phase_profile_read(clear=True)
ref_out, ref = oracle.run_case(c)
assert_parity(out, grads, ref_out, ref, "profiling build")
for d in (0, 1):
    ctas = [q for q in data[d] if q[4] > 0]
    assert ctas, d
    for q in ctas:
        assert q[4] >= 1 and q[5] == q[4] - 1, (d, q)   # one barrier between microsteps
        assert 0 < q[0] <= q[1], (d, q)                  # part A within part A + sync
        assert q[2] > 0 and (q[4] < 2 or q[3] > 0), (d, q)
    assert max(q[4] for q in ctas) >= S, (d, S)
    assert sum(q[7] & 0xffffffff for q in ctas) == c["E"], d   # the pieces cover every edge
again = _ck.ck_phase_profile_read(clear=False)
assert all(v == 0 for dd in again for q in dd for v in q)     # cleared by the read before
print("profile ok")
'''


def test_profiling_build_counts_and_parity():
    env = dict(os.environ)
    env["CK_LIBRARY_VARIANT"] = "prof"
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "profile ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


RUN = r'''
import sys
sys.path.insert(0, "tests")
import numpy as np
import workloads
from gpu_helpers import run_gpu
c = workloads.small(922, 700, 30000, 10, 32, 3, 2, hub_deg=9000, dup_frac=0.05)
out, grads = run_gpu(c)
np.savez(sys.argv[1], out=out, **grads)
print("saved")
'''


def test_every_build_gives_the_same_bits(tmp_path):
    """The bounds-checked and profiling builds compute exactly what the
    ordinary build does (their extra code only checks indices or reads the
    clock): outputs and all five gradients equal bit for bit."""
    import numpy as np
    res = {}
    for variant in ("", "bounds", "prof"):
        env = dict(os.environ)
        env["CK_LIBRARY_VARIANT"] = variant
        path = str(tmp_path / f"run_{variant or 'plain'}.npz")
        r = subprocess.run([sys.executable, "-c", RUN, path], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=600)
        assert r.returncode == 0 and "saved" in r.stdout, (variant, r.stdout[-2000:] + r.stderr[-2000:])
        res[variant] = np.load(path)
    for variant in ("bounds", "prof"):
        for k in res[""].files:
            np.testing.assert_array_equal(res[variant][k], res[""][k], err_msg=f"{variant} {k}")
