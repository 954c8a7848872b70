"""Shared pieces of the GPU parity tests: run a workload through the C ABI and
compare with the oracle under the stated tolerances."""
import numpy as np
import torch

# states: max |gpu - oracle| <= 1e-5 (states are bounded by 1);
# gradients: max |gpu - oracle| / max |oracle| <= 1e-4, per tensor.
STATE_TOL = 1e-5
GRAD_TOL = 1e-4
GRAD_KEYS = ("dw", "dleak", "dbias", "ddrives", "dstate0")


def to_dev(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def make_graph(c, tiling=None):
    """The graph of case c; with its shared-memory tilings when `tiling`, by
    default whenever the tiled kernels are switched on (CK_OPT_TILED), so that
    a test selecting them runs them where the graph allows."""
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    if tiling is None:
        tiling = _ck.ck_get_option(_ck.OPT_TILED) != 0
    return pkg.SparseGraph(to_dev(c["src"]), to_dev(c["dst"]), c["N"], to_dev(c["input_nodes"]),
                           tiling=tiling)


def run_gpu(c, M=None, graph=None, dout=None):
    """Forward and backward through ck_forward / ck_backward.  Returns numpy
    (out[T,B,N], dict of the five gradients)."""
    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    M = c["M"] if M is None else M
    g = graph or make_graph(c)
    w, leak, bias = to_dev(c["w"]), to_dev(c["leak"]), to_dev(c["bias"])
    drives, state0 = to_dev(c["drives"]), to_dev(c["state0"])
    B, T = c["state0"].shape[0], c["drives"].shape[0]
    out, saved, scratch = pkg.forward(g, w, leak, bias, drives, state0, M)
    _ck.ck_query_status(scratch)
    d = to_dev(c["dout"] if dout is None else dout)
    grads = pkg.backward(g, w, leak, B, T, M, saved, d, scratch)
    _ck.ck_query_status(scratch)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy().astype(np.float64) for k, v in zip(GRAD_KEYS, grads)}
    return out.cpu().numpy().astype(np.float64), res


def rel_err(got, ref):
    scale = np.abs(ref).max(initial=0.0)
    diff = np.abs(got - ref).max(initial=0.0)
    if scale == 0.0:
        return diff
    return diff / scale


def assert_parity(out, grads, ref_out, ref_grads, what=""):
    e = np.abs(out - ref_out).max(initial=0.0)
    assert e <= STATE_TOL, f"{what} states: max abs err {e:.3e}"
    for k in GRAD_KEYS:
        r = rel_err(grads[k], ref_grads[k])
        assert r <= GRAD_TOL, f"{what} {k}: normalised err {r:.3e}"
