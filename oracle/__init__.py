"""The oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU statement of what the library computes, used only by
`tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`.
The CUDA library never imports or calls it.  It shares no code with the CUDA
path: the recurrence and its backward are in `ck_oracle.c` (fp64, loops over
the caller's edge order); the compressed-row layouts the library must build are
defined here by a stable sort, ties kept in ascending edge id.

Sources (connectome-kernels page): intro (update equations, sparse W with one
scalar per edge, drive only at input nodes); "Use" (argument shapes, edge
direction src -> dst, edge parameters in the caller's order while the internal
compressed-row permutation stays invisible); "Design notes" (transposed
compressed rows for the state gradient).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ck_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libck_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ck_oracle.c with gcc -O2 (no fast-math) into oracle/_build/."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math"]
        # OpenMP serves only oracle_step_columns (batch columns on several
        # cores); without it that function runs on one thread
        if subprocess.call(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"],
                           stderr=subprocess.DEVNULL) != 0:
            subprocess.check_call(base + ["-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_forward.argtypes = [i64, i64, p, p, p, p, p, i64, p, p, p,
                                       i64, i64, i64, p, p, p]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [i64, i64, p, p, p, p, i64, p, i64, i64,
                                        i64, p, p, p, p, p, p, p, p]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_step_columns.argtypes = [i64, i64, p, p, p, p, p, i64, p, p, p, p,
                                            i64, i64, i64, ctypes.c_int, p, p, p, p, p, p]
        lib.oracle_step_columns.restype = ctypes.c_int
        lib.oracle_threads_available.argtypes = []
        lib.oracle_threads_available.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _i64(x):
    return np.ascontiguousarray(x, dtype=np.int64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def forward(N, src, dst, w, leak, bias, input_nodes, drives, state0, M):
    """Run the recurrence.  Returns (out[T,B,N], hprev[S,B,N], pre[S,B,N]).

    hprev[s] is the state entering microstep s; pre[s] the pre-activation.
    """
    src, dst, input_nodes = _i64(src), _i64(dst), _i64(input_nodes)
    w, leak, bias = _f64(w), _f64(leak), _f64(bias)
    drives, state0 = _f64(drives), _f64(state0)
    T, n_in, B = drives.shape
    assert state0.shape == (B, N) and n_in == input_nodes.size
    S = T * M
    out = np.empty((T, B, N))
    hprev = np.empty((S, B, N))
    pre = np.empty((S, B, N))
    rc = _load().oracle_forward(N, src.size, _ptr(src), _ptr(dst), _ptr(w), _ptr(leak),
                                _ptr(bias), n_in, _ptr(input_nodes), _ptr(drives),
                                _ptr(state0), B, T, M, _ptr(out), _ptr(hprev), _ptr(pre))
    if rc != 0:
        raise MemoryError("oracle_forward could not allocate")
    return out, hprev, pre


def backward(N, src, dst, w, leak, input_nodes, hprev, pre, dout, M):
    """VJP of L = sum_t <dout[t], out[t]>.

    Returns dict(dw[E], dleak[N], dbias[N], ddrives[T,n_in,B], dstate0[B,N]).
    """
    src, dst, input_nodes = _i64(src), _i64(dst), _i64(input_nodes)
    w, leak = _f64(w), _f64(leak)
    hprev, pre, dout = _f64(hprev), _f64(pre), _f64(dout)
    T, B, _ = dout.shape
    n_in = input_nodes.size
    E = src.size
    dw = np.empty(E)
    dleak = np.empty(N)
    dbias = np.empty(N)
    ddrives = np.empty((T, n_in, B))
    dstate0 = np.empty((B, N))
    rc = _load().oracle_backward(N, E, _ptr(src), _ptr(dst), _ptr(w), _ptr(leak), n_in,
                                 _ptr(input_nodes), B, T, M, _ptr(hprev), _ptr(pre),
                                 _ptr(dout), _ptr(dw), _ptr(dleak), _ptr(dbias),
                                 _ptr(ddrives), _ptr(dstate0))
    if rc != 0:
        raise MemoryError("oracle_backward could not allocate")
    return dict(dw=dw, dleak=dleak, dbias=dbias, ddrives=ddrives, dstate0=dstate0)


def run_case(case: dict, M: int | None = None, batch_cols=None):
    """Forward and backward of a workload dict from `workloads`.

    batch_cols restricts the run to some batch columns (they are independent
    sequences); the edge, leak and bias gradients are then those of the loss
    restricted to these columns.
    """
    M = case["M"] if M is None else M
    drives, state0, dout = case["drives"], case["state0"], case["dout"]
    if batch_cols is not None:
        cols = np.asarray(batch_cols)
        drives, state0, dout = drives[:, :, cols], state0[cols], dout[:, cols]
    out, hprev, pre = forward(case["N"], case["src"], case["dst"], case["w"], case["leak"],
                              case["bias"], case["input_nodes"], drives, state0, M)
    grads = backward(case["N"], case["src"], case["dst"], case["w"], case["leak"],
                     case["input_nodes"], hprev, pre, dout, M)
    return out, grads


def threads_available() -> int:
    """Cores the OpenMP step may use (1 when built without OpenMP)."""
    return int(_load().oracle_threads_available())


def step_columns(case: dict, threads: int, M: int | None = None):
    """One whole step (forward and backward) of a workload dict, its batch
    columns spread over `threads` threads.  Same results as run_case up to
    the grouping of the sums over columns of dw, dleak and dbias (per thread,
    then over threads in order).  Returns (out, grads) like run_case."""
    M = case["M"] if M is None else M
    N = case["N"]
    src, dst, inp = _i64(case["src"]), _i64(case["dst"]), _i64(case["input_nodes"])
    w, leak, bias = _f64(case["w"]), _f64(case["leak"]), _f64(case["bias"])
    drives, state0, dout = _f64(case["drives"]), _f64(case["state0"]), _f64(case["dout"])
    T, n_in, B = drives.shape
    E = src.size
    out = np.empty((T, B, N))
    g = dict(dw=np.empty(E), dleak=np.empty(N), dbias=np.empty(N),
             ddrives=np.empty((T, n_in, B)), dstate0=np.empty((B, N)))
    rc = _load().oracle_step_columns(N, E, _ptr(src), _ptr(dst), _ptr(w), _ptr(leak),
                                     _ptr(bias), n_in, _ptr(inp), _ptr(drives), _ptr(state0),
                                     _ptr(dout), B, T, M, int(threads), _ptr(out),
                                     _ptr(g["dw"]), _ptr(g["dleak"]), _ptr(g["dbias"]),
                                     _ptr(g["ddrives"]), _ptr(g["dstate0"]))
    if rc != 0:
        raise MemoryError("oracle_step_columns could not allocate")
    return out, g


def csr(N: int, key, other):
    """Compressed rows keyed by `key`: a stable sort, ties in ascending edge id.

    Returns (row_ptr[N+1], col[E] = other[perm], perm[E]) as int32, where
    row_ptr is the exclusive prefix sum of the key counts and perm[k] is the
    caller's id of the k-th edge in row order.
    """
    key = _i64(key)
    perm = np.argsort(key, kind="stable")
    counts = np.bincount(key, minlength=N)
    row_ptr = np.zeros(N + 1, np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    return (row_ptr.astype(np.int32), _i64(other)[perm].astype(np.int32),
            perm.astype(np.int32))


def graph_layout(N: int, src, dst, input_nodes):
    """Everything the library's graph build must reproduce bit for bit.

    Forward rows are keyed by dst (node i sums over its in-edges), transposed
    rows by src; slot[i] = k when input_nodes[k] = i, else -1.
    """
    row_ptr, col, perm = csr(N, dst, src)
    rowT_ptr, colT, permT = csr(N, src, dst)
    slot = np.full(N, -1, np.int32)
    slot[_i64(input_nodes)] = np.arange(len(input_nodes), dtype=np.int32)
    return dict(row_ptr=row_ptr, col=col, perm=perm, rowT_ptr=rowT_ptr, colT=colT,
                permT=permT, slot=slot)


def adam_update(param, grad, m, v, step: int, lr: float, beta1: float, beta2: float, eps: float):
    """One Adam step in fp64 (Kingma and Ba, "Adam: A Method for Stochastic
    Optimization", Algorithm 1), the optional optimizer of a captured training
    step (TrainKernel page: the captured step holds the parameter update).
    `step` is t >= 1.  Returns (param, m, v) after the step:
        m <- beta1 m + (1 - beta1) g;   v <- beta2 v + (1 - beta2) g^2
        param <- param - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
    """
    p = np.asarray(param, np.float64)
    g = np.asarray(grad, np.float64)
    m = beta1 * np.asarray(m, np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, np.float64) + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** step)
    vhat = v / (1.0 - beta2 ** step)
    return p - lr * mhat / (np.sqrt(vhat) + eps), m, v
