"""Pins for the oracle (CPU only).

The oracle is checked here against things other than itself: hand-derived
layouts, closed forms of special cases, a dense-matrix brute force, central
finite differences of its own forward (for the backward), and invariants of
the recurrence.  The recurrence is the one of the connectome-kernels page
(intro: proposal = tanh(W h + drive + bias); h <- (1-leak) h + leak*proposal,
repeated `microsteps` times per input step).
"""
import math

import numpy as np
import pytest

import workloads
from golden_io import read_cases


def _case(seed=7, N=12, E=40, n_in=3, B=3, T=3, M=2, **kw):
    return workloads.small(seed, N, E, n_in, B, T, M, **kw)


def _fwd(oracle, c, **over):
    d = dict(c)
    d.update(over)
    return oracle.forward(d["N"], d["src"], d["dst"], d["w"], d["leak"], d["bias"],
                          d["input_nodes"], d["drives"], d["state0"], d["M"])


def _bwd(oracle, c, **over):
    d = dict(c)
    d.update(over)
    out, hprev, pre = _fwd(oracle, d)
    g = oracle.backward(d["N"], d["src"], d["dst"], d["w"], d["leak"], d["input_nodes"],
                        hprev, pre, d["dout"], d["M"])
    return out, g


# --------------------------------------------------------------------------
# graph layout: stable compressed rows, hand-derived expectations
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", read_cases("csr_tiny.txt"), ids=lambda c: c["name"])
def test_layout_matches_hand_derived(oracle_lib, case):
    lay = oracle_lib.graph_layout(case["N"], case["src"], case["dst"], case["input_nodes"])
    for k in ("row_ptr", "col", "perm", "rowT_ptr", "colT", "permT", "slot"):
        np.testing.assert_array_equal(lay[k].astype(np.int64), case[k], err_msg=k)


def test_layout_ties_keep_edge_order(oracle_lib):
    # all edges share one destination: rows must keep the caller's order
    N, E = 6, 50
    rng = np.random.default_rng(3)
    src = rng.integers(0, N, E)
    dst = np.full(E, 2)
    lay = oracle_lib.graph_layout(N, src, dst, [0])
    np.testing.assert_array_equal(lay["perm"], np.arange(E))
    # transposed rows: within each source, ascending edge id
    for j in range(N):
        seg = lay["permT"][lay["rowT_ptr"][j]:lay["rowT_ptr"][j + 1]]
        assert np.all(np.diff(seg) > 0) and np.all(src[seg] == j)


# --------------------------------------------------------------------------
# forward: closed forms
# --------------------------------------------------------------------------

def test_leak_zero_keeps_state(oracle_lib):
    c = _case()
    out, _, _ = _fwd(oracle_lib, c, leak=np.zeros(c["N"], np.float32))
    for t in range(c["T"]):
        np.testing.assert_array_equal(out[t], c["state0"].astype(np.float64))


@pytest.mark.parametrize("M", [1, 2, 3])
def test_no_edges_relaxes_geometrically(oracle_lib, M):
    # W = 0 and a drive held constant over the input steps:
    # out[t] = p* + (1-leak)^((t+1) M) (h0 - p*), p* = tanh(drive + bias)
    c = _case(M=M, T=4)
    N, B, T = c["N"], c["B"], c["T"]
    drv = np.repeat(c["drives"][:1], T, axis=0)
    out, _, _ = _fwd(oracle_lib, c, w=np.zeros(c["E"], np.float32), drives=drv)
    d = np.zeros((B, N))
    for k, node in enumerate(c["input_nodes"]):
        d[:, node] = drv[0, k, :]
    h0 = c["state0"].astype(np.float64)
    lam = c["leak"].astype(np.float64)
    beta = c["bias"].astype(np.float64)
    for t in range(T):
        for b in range(B):
            for i in range(N):
                p = math.tanh(d[b, i] + beta[i])
                want = p + (1.0 - lam[i]) ** ((t + 1) * M) * (h0[b, i] - p)
                assert abs(out[t, b, i] - want) < 1e-13


@pytest.mark.parametrize("M", [1, 3])
def test_self_loops_only_is_a_scalar_recursion_per_node(oracle_lib, M):
    # With every edge a self-loop, W is diagonal (repeated loops add) and each
    # node follows its own scalar recursion, microstep by microstep:
    #   h <- (1 - leak_i) h + leak_i tanh(W_ii h + drive_i(t) + bias_i)
    c = _case(seed=31, N=40, E=120, n_in=5, B=3, T=3, M=M, loops_only=True)
    N, B, T = c["N"], c["B"], c["T"]
    assert np.all(c["src"] == c["dst"])
    out, _, _ = _fwd(oracle_lib, c)
    wdiag = [0.0] * N
    for s_, v in zip(c["src"], c["w"]):
        wdiag[int(s_)] += float(v)
    slot = {int(node): k for k, node in enumerate(c["input_nodes"])}
    for b in range(B):
        for i in range(N):
            h = float(c["state0"][b, i])
            lam, beta = float(c["leak"][i]), float(c["bias"][i])
            for t in range(T):
                d = float(c["drives"][t, slot[i], b]) if i in slot else 0.0
                for _ in range(M):
                    h = (1.0 - lam) * h + lam * math.tanh(wdiag[i] * h + d + beta)
                assert abs(out[t, b, i] - h) < 1e-13, (b, i, t)


@pytest.mark.parametrize("M", [1, 2, 3])
def test_chain_propagates_one_node_per_microstep(oracle_lib, M):
    # Chain 0 -> 1 -> ... -> N-1, unit weights, leak 1, bias 0, state0 0, drive
    # d only at node 0.  With a synchronous update node k first moves at
    # microstep k, and then holds the (k+1)-fold iterated tanh of d.  A swapped
    # edge direction or an in-place sweep breaks this.
    N, T, B = 7, 3, 2
    src = np.arange(N - 1)
    dst = np.arange(1, N)
    dval = np.array([0.8, -1.3])
    drives = np.tile(dval[None, None, :], (T, 1, 1)).astype(np.float32)
    out, _, _ = oracle_lib.forward(N, src, dst, np.ones(N - 1, np.float32),
                                   np.ones(N, np.float32), np.zeros(N, np.float32), [0],
                                   drives, np.zeros((B, N), np.float32), M)
    for t in range(T):
        s = (t + 1) * M - 1  # last microstep of step t
        for b in range(B):
            v = float(np.float32(dval[b]))
            for k in range(N):
                if k > s:
                    assert out[t, b, k] == 0.0
                else:
                    want = v
                    for _ in range(k + 1):
                        want = math.tanh(want)
                    assert abs(out[t, b, k] - want) < 1e-14


def test_single_edge_by_hand(oracle_lib):
    # 2 nodes, one edge 0 -> 1.  One microstep, written out term by term.
    w, l0, l1, b0, b1, h0, h1, d = 0.7, 0.25, 0.6, 0.1, -0.2, 0.3, -0.4, 0.9
    f = np.float32
    out, _, _ = oracle_lib.forward(2, [0], [1], np.array([w], f), np.array([l0, l1], f),
                                   np.array([b0, b1], f), [0], np.array([[[d]]], f),
                                   np.array([[h0, h1]], f), 1)
    W, L0, L1, B0, B1, H0, H1, D = (float(f(x)) for x in (w, l0, l1, b0, b1, h0, h1, d))
    want0 = (1 - L0) * H0 + L0 * math.tanh(D + B0)        # node 0: drive, no in-edge
    want1 = (1 - L1) * H1 + L1 * math.tanh(W * H0 + B1)    # node 1: edge from node 0
    assert abs(out[0, 0, 0] - want0) < 1e-15
    assert abs(out[0, 0, 1] - want1) < 1e-15


# --------------------------------------------------------------------------
# dense-matrix brute force (forward and backward)
# --------------------------------------------------------------------------

def _dense(c):
    N = c["N"]
    W = np.zeros((N, N))
    np.add.at(W, (c["dst"], c["src"]), c["w"].astype(np.float64))
    return W


def _dense_forward(c):
    W = _dense(c)
    lam = c["leak"].astype(np.float64)
    beta = c["bias"].astype(np.float64)
    T, M, B, N = c["T"], c["M"], c["B"], c["N"]
    H = c["state0"].astype(np.float64)          # [B, N]
    outs, hs, As = [], [], []
    for t in range(T):
        D = np.zeros((B, N))
        D[:, c["input_nodes"]] = c["drives"][t].T.astype(np.float64)
        for _ in range(M):
            A = H @ W.T + D + beta
            hs.append(H)
            As.append(A)
            H = (1 - lam) * H + lam * np.tanh(A)
        outs.append(H)
    return np.stack(outs), hs, As, W


def _dense_backward(c):
    out, hs, As, W = _dense_forward(c)
    lam = c["leak"].astype(np.float64)
    T, M = c["T"], c["M"]
    dout = c["dout"].astype(np.float64)
    G = np.zeros_like(hs[0])
    dW = np.zeros_like(W)
    dlam = np.zeros(c["N"])
    dbeta = np.zeros(c["N"])
    ddrv = np.zeros(c["drives"].shape)
    for s in reversed(range(T * M)):
        t, m = divmod(s, M)
        if m == M - 1:
            G = G + dout[t]
        P = np.tanh(As[s])
        dA = G * lam * (1 - P * P)
        dlam += (G * (P - hs[s])).sum(0)
        dbeta += dA.sum(0)
        ddrv[t] += dA[:, c["input_nodes"]].T
        dW += dA.T @ hs[s]
        G = G * (1 - lam) + dA @ W
    return dict(dw=dW[c["dst"], c["src"]], dleak=dlam, dbias=dbeta, ddrives=ddrv, dstate0=G)


@pytest.mark.parametrize("seed,kw", [
    (11, dict(N=16, E=60, dup_frac=0.2)),
    (12, dict(N=30, E=200, B=4, T=2, M=3, hub_deg=50)),
    (13, dict(N=9, E=0, B=2)),
    (14, dict(N=40, E=300, B=5, T=4, M=1, self_loops=False)),
])
def test_dense_bruteforce(oracle_lib, seed, kw):
    c = _case(seed=seed, **kw)
    out, g = _bwd(oracle_lib, c)
    dout, _, _, _ = _dense_forward(c)
    np.testing.assert_allclose(out, dout, rtol=0, atol=1e-12)
    dg = _dense_backward(c)
    for k in dg:
        scale = max(1.0, np.abs(dg[k]).max(initial=0.0))
        assert np.abs(g[k] - dg[k]).max(initial=0.0) <= 1e-12 * scale, k


# --------------------------------------------------------------------------
# backward: central finite differences of the oracle's own forward
# --------------------------------------------------------------------------

def _loss(oracle, c, **over):
    out, _, _ = _fwd(oracle, c, **over)
    return float((out * c["dout"].astype(np.float64)).sum())


@pytest.mark.parametrize("seed,kw", [
    (21, dict(N=8, E=24, n_in=2, B=1, T=2, M=1, dup_frac=0.25)),
    (22, dict(N=10, E=40, n_in=3, B=3, T=3, M=2, dup_frac=0.1)),
    (23, dict(N=12, E=30, n_in=2, B=3, T=2, M=3, hub_deg=10)),
])
def test_backward_matches_finite_differences(oracle_lib, seed, kw):
    c = _case(seed=seed, **kw)
    # fp64 copies of the inputs so perturbations are not rounded to fp32
    c = {k: (v.astype(np.float64) if isinstance(v, np.ndarray) and v.dtype == np.float32 else v)
         for k, v in c.items()}
    _, g = _bwd(oracle_lib, c)
    eps = 1e-6
    for name, key in (("w", "dw"), ("leak", "dleak"), ("bias", "dbias"),
                      ("drives", "ddrives"), ("state0", "dstate0")):
        base = c[name]
        fd = np.zeros(base.shape)
        for idx in np.ndindex(base.shape):
            up = base.copy()
            dn = base.copy()
            up[idx] += eps
            dn[idx] -= eps
            fd[idx] = (_loss(oracle_lib, c, **{name: up}) - _loss(oracle_lib, c, **{name: dn})) / (2 * eps)
        scale = max(np.abs(g[key]).max(), 1e-3)
        err = np.abs(fd - g[key]).max() / scale
        assert err < 1e-7, (key, err)


# --------------------------------------------------------------------------
# backward: closed forms
# --------------------------------------------------------------------------

def test_backward_leak_zero(oracle_lib):
    # leak = 0: the state never moves, so dstate0 = sum_t dout[t], and nothing
    # flows into w, bias or drives; dleak_i = sum_{t,m,b} G_t (tanh(W h0 + d_t + b) - h0)
    # with G_t = sum_{t' >= t} dout[t'].
    c = _case(seed=31, N=14, E=50, B=3, T=3, M=2)
    c["leak"] = np.zeros(c["N"], np.float32)
    _, g = _bwd(oracle_lib, c)
    dout = c["dout"].astype(np.float64)
    np.testing.assert_allclose(g["dstate0"], dout.sum(0), rtol=0, atol=1e-14)
    for k in ("dw", "dbias", "ddrives"):
        assert np.all(g[k] == 0.0), k
    W = _dense(c)
    h0 = c["state0"].astype(np.float64)
    want = np.zeros(c["N"])
    for t in range(c["T"]):
        D = np.zeros_like(h0)
        D[:, c["input_nodes"]] = c["drives"][t].T
        P = np.tanh(h0 @ W.T + D + c["bias"].astype(np.float64))
        Gt = dout[t:].sum(0)
        want += c["M"] * (Gt * (P - h0)).sum(0)
    np.testing.assert_allclose(g["dleak"], want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("M", [1, 2, 3])
def test_backward_no_edges_scalar_closed_forms(oracle_lib, M):
    # W = 0, constant drive, r = 1 - leak, p* = tanh(d + bias):
    #   d out[t] / d h0        = r^((t+1)M)
    #   d out[t] / d bias      = (1 - r^((t+1)M)) (1 - p*^2)
    #   d out[t] / d drive[t'] = r^((t-t')M) (1 - r^M) (1 - p*^2),  t' <= t
    c = _case(seed=41, N=6, E=10, n_in=2, B=2, T=3, M=M)
    T = c["T"]
    c["w"] = np.zeros(c["E"], np.float32)
    c["drives"] = np.repeat(c["drives"][:1], T, axis=0)
    lam = c["leak"].astype(np.float64)
    beta = c["bias"].astype(np.float64)
    node = int(c["input_nodes"][1])
    b = 1
    d = float(c["drives"][0, 1, b])
    p = math.tanh(d + beta[node])
    r = 1.0 - lam[node]
    for t in range(T):
        dout = np.zeros_like(c["dout"])
        dout[t, b, node] = 1.0
        _, g = _bwd(oracle_lib, c, dout=dout)
        assert abs(g["dstate0"][b, node] - r ** ((t + 1) * M)) < 1e-14
        assert abs(g["dbias"][node] - (1 - r ** ((t + 1) * M)) * (1 - p * p)) < 1e-14
        for tp in range(T):
            want = r ** ((t - tp) * M) * (1 - r ** M) * (1 - p * p) if tp <= t else 0.0
            assert abs(g["ddrives"][tp, 1, b] - want) < 1e-14
        # nothing else receives gradient
        mask = np.ones_like(g["dstate0"], bool)
        mask[b, node] = False
        assert np.all(g["dstate0"][mask] == 0.0)
        # edge values only receive gradient on edges into the probed node
        assert np.all(g["dw"][c["dst"] != node] == 0.0)


def test_backward_linear_in_dout(oracle_lib):
    c = _case(seed=51, N=15, E=60, B=2, T=3, M=2)
    rng = np.random.default_rng(5)
    d1 = rng.normal(size=c["dout"].shape)
    d2 = rng.normal(size=c["dout"].shape)
    _, g1 = _bwd(oracle_lib, c, dout=d1)
    _, g2 = _bwd(oracle_lib, c, dout=d2)
    _, g12 = _bwd(oracle_lib, c, dout=d1 + 2.0 * d2)
    for k in g1:
        np.testing.assert_allclose(g12[k], g1[k] + 2.0 * g2[k], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_state_stays_in_unit_ball(oracle_lib):
    c = _case(seed=61, N=50, E=400, B=4, T=6, M=3, w_scale=3.0)
    out, hprev, _ = _fwd(oracle_lib, c)
    assert np.abs(c["state0"]).max() < 1
    assert np.abs(out).max() <= 1.0 and np.abs(hprev).max() <= 1.0


def test_relabelling_permutes_everything(oracle_lib):
    c = _case(seed=71, N=20, E=90, B=2, T=2, M=2, dup_frac=0.1)
    out, g = _bwd(oracle_lib, c)
    rng = np.random.default_rng(9)
    pi = rng.permutation(c["N"])          # old id i -> new id pi[i]
    inv = np.argsort(pi)
    r = dict(c)
    r["src"], r["dst"], r["input_nodes"] = pi[c["src"]], pi[c["dst"]], pi[c["input_nodes"]]
    r["leak"], r["bias"] = c["leak"][inv], c["bias"][inv]
    r["state0"], r["dout"] = c["state0"][:, inv], c["dout"][:, :, inv]
    out_r, g_r = _bwd(oracle_lib, r)
    np.testing.assert_allclose(out_r, out[:, :, inv], rtol=0, atol=1e-14)
    np.testing.assert_allclose(g_r["dw"], g["dw"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g_r["dleak"], g["dleak"][inv], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g_r["dstate0"], g["dstate0"][:, inv], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g_r["ddrives"], g["ddrives"], rtol=1e-12, atol=1e-14)


def test_edge_order_and_splitting(oracle_lib):
    c = _case(seed=81, N=18, E=70, B=3, T=2, M=2)
    out, g = _bwd(oracle_lib, c)
    # shuffled edge order: same outputs, permuted edge gradient
    q = np.random.default_rng(4).permutation(c["E"])
    s = dict(c, src=c["src"][q], dst=c["dst"][q], w=c["w"][q])
    out_s, g_s = _bwd(oracle_lib, s)
    np.testing.assert_allclose(out_s, out, rtol=0, atol=1e-14)
    np.testing.assert_allclose(g_s["dw"], g["dw"][q], rtol=1e-12, atol=1e-14)
    # split edge 5 into two parallel copies whose values add up to the original
    w64 = c["w"].astype(np.float64)
    w1 = 0.3 * w64[5]
    sp = dict(c, src=np.append(c["src"], c["src"][5]), dst=np.append(c["dst"], c["dst"][5]),
              w=np.append(np.where(np.arange(c["E"]) == 5, w64[5] - w1, w64), w1), E=c["E"] + 1)
    for k in ("leak", "bias", "drives", "state0", "dout"):
        sp[k] = c[k].astype(np.float64)
    base = {k: (v.astype(np.float64) if isinstance(v, np.ndarray) and v.dtype == np.float32 else v)
            for k, v in c.items()}
    out_b, g_b = _bwd(oracle_lib, base)
    out_p, g_p = _bwd(oracle_lib, sp)
    np.testing.assert_allclose(out_p, out_b, rtol=0, atol=1e-14)
    assert abs(g_p["dw"][5] - g_b["dw"][5]) < 1e-13
    assert abs(g_p["dw"][-1] - g_b["dw"][5]) < 1e-13


# --------------------------------------------------------------------------
# run_case(batch_cols=...): the column-restricted run the full-size parity
# tests compare against.  Batch columns are independent sequences (intro: the
# recurrence runs per sample), so restricting to some columns must give those
# columns of the full run, and the shared-parameter gradients must be the full
# run's with dOut zero outside them.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("cols", [[1, 4], [0], [5, 2, 3]])
def test_run_case_batch_cols(oracle_lib, cols):
    c = _case(seed=31, N=14, E=60, n_in=4, B=6, T=3, M=2)
    out_c, g_c = oracle_lib.run_case(c, batch_cols=cols)
    out_f, g_f = oracle_lib.run_case(c)
    np.testing.assert_allclose(out_c, out_f[:, cols], rtol=0, atol=1e-15)
    np.testing.assert_allclose(g_c["ddrives"], g_f["ddrives"][:, :, cols], rtol=0, atol=1e-15)
    np.testing.assert_allclose(g_c["dstate0"], g_f["dstate0"][cols], rtol=0, atol=1e-15)
    masked = dict(c)
    keep = np.zeros(c["B"], bool)
    keep[cols] = True
    masked["dout"] = np.where(keep[None, :, None], c["dout"], 0.0)
    _, g_m = oracle_lib.run_case(masked)
    for k in ("dw", "dleak", "dbias"):
        np.testing.assert_allclose(g_c[k], g_m[k], rtol=1e-13, atol=1e-15, err_msg=k)
        # and the mask matters: the unmasked full run differs
        assert np.abs(g_f[k] - g_c[k]).max() > 1e-6, k


# --------------------------------------------------------------------------
# step_columns: the multi-core statement of one step used for the timed CPU
# baseline.  It must agree with the single-thread oracle (pinned above) for
# every thread count, differing only in the grouping of the column sums.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("threads", [1, 2, 3, 4, 16])
def test_step_columns_matches_single_thread(oracle_lib, threads):
    c = _case(seed=41, N=20, E=90, n_in=5, B=7, T=3, M=2, hub_deg=30)
    out_r, g_r = oracle_lib.run_case(c)
    out_p, g_p = oracle_lib.step_columns(c, threads)
    assert np.array_equal(out_p, out_r)
    for k in ("ddrives", "dstate0"):
        assert np.array_equal(g_p[k], g_r[k]), k
    for k in ("dw", "dleak", "dbias"):
        scale = np.abs(g_r[k]).max()
        assert np.abs(g_p[k] - g_r[k]).max() <= 1e-12 * scale, k
    # a second run with the same thread count repeats every bit
    out_q, g_q = oracle_lib.step_columns(c, threads)
    assert all(np.array_equal(g_q[k], g_p[k]) for k in g_p)


# --------------------------------------------------------------------------
# the optional Adam update of a captured training step
# --------------------------------------------------------------------------

def test_adam_first_step_closed_form():
    # from m = v = 0 the bias corrections make m_hat = g and v_hat = g^2, so
    # the first step moves every parameter by lr g / (|g| + eps)
    import oracle
    rng = np.random.default_rng(5)
    p, g = rng.normal(size=50), rng.normal(size=50)
    lr, eps = 0.01, 1e-8
    p1, m1, v1 = oracle.adam_update(p, g, np.zeros(50), np.zeros(50), 1, lr, 0.9, 0.999, eps)
    np.testing.assert_allclose(p1, p - lr * g / (np.abs(g) + eps), rtol=0, atol=1e-15)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-12)


def test_adam_constant_gradient_closed_form():
    # with the same gradient every step, m_t = (1 - beta1^t) g and
    # v_t = (1 - beta2^t) g^2 exactly, so every step moves by lr g / (|g| + eps)
    import oracle
    rng = np.random.default_rng(6)
    p0, g = rng.normal(size=20), rng.normal(size=20)
    p, m, v = p0.copy(), np.zeros(20), np.zeros(20)
    lr, eps, b1, b2 = 0.003, 1e-6, 0.8, 0.95
    for t in range(1, 26):
        p, m, v = oracle.adam_update(p, g, m, v, t, lr, b1, b2, eps)
        np.testing.assert_allclose(m, (1 - b1 ** t) * g, rtol=1e-12)
        np.testing.assert_allclose(p, p0 - t * lr * g / (np.abs(g) + eps), rtol=0, atol=1e-12)
