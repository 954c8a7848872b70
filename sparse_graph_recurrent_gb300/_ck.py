"""ctypes binding of libck's C ABI (include/ck.h): argument marshalling only.

Every function here has the name of the C entry point it calls and takes torch
CUDA tensors in place of raw device pointers.  All computation happens in the
library's CUDA kernels; if the library cannot be built or loaded this module
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

CK_OK = 0
STATUS = {0: "CK_OK", 1: "CK_ERR_INVALID_ARG", 2: "CK_ERR_CUDA", 3: "CK_ERR_OUT_OF_MEMORY",
          4: "CK_ERR_TIMEOUT", 5: "CK_ERR_WORKSPACE", 6: "CK_ERR_INTERNAL",
          7: "CK_ERR_UNSUPPORTED"}
(OPT_PERSISTENT, OPT_BARRIER_TIMEOUT_NS, OPT_TEST_BARRIER_EXTRA, OPT_GRAPH_IN_SMEM,
 OPT_RECOMPUTE_STEPS, OPT_ROWS_IN_SMEM, OPT_TEST_BOUNDS_PROBE, OPT_TILED) = range(8)
GRAPH_EDGES_IN_HOST_MEMORY, GRAPH_TILING = 1, 2  # ck_graph_flag
# ck_barrier_scheme (ck_probe_grid_barrier)
(BARRIER_COUNTER, BARRIER_COUNTER_RETURNING, BARRIER_COUNTER_RELAXED, BARRIER_FLAG,
 BARRIER_FLAGS8, BARRIER_CLUSTER_SYNC, BARRIER_CLUSTER_MBARRIER) = range(7)
PROBE_BARRIER_WORDS = 16384
PHASE_PROFILE_CTAS, PHASE_PROFILE_WORDS = 1024, 8  # ck_phase_profile_read

_lib = None


class CKError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS.get(status, str(status))


def library_variant():
    """The library variant this process loads: None (libck.so), "bounds"
    (libck_bounds.so, the bounds-checked build) or "prof" (libck_prof.so, with
    the phase profile), from CK_LIBRARY_VARIANT."""
    return os.environ.get("CK_LIBRARY_VARIANT") or None


def library_path() -> str:
    return _build.lib_path(library_variant())


def load() -> ctypes.CDLL:
    """Load the library, building it with nvcc first if it is missing or stale."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build(variant=library_variant())
    if not os.path.exists(path):
        raise ImportError(f"libck.so not found at {path}")
    lib = ctypes.CDLL(path)
    p, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    psz = ctypes.POINTER(ctypes.c_size_t)
    pi64 = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "ck_graph_create": [p, p, i64, i64, p, i64, p, ctypes.POINTER(p)],
        "ck_graph_create_flags": [p, p, i64, i64, p, i64, ctypes.c_uint32, p, ctypes.POINTER(p)],
        "ck_graph_destroy": [p],
        "ck_graph_info": [p, pi64, pi64, pi64],
        "ck_graph_memory": [p, psz, psz],
        "ck_graph_tiling": [p, ctypes.c_int, pi64],
        "ck_graph_export_tiling": [p, ctypes.c_int, p, p, p, p, p, p],
        "ck_graph_export": [p, p, p, p, p, p, p, p, p],
        "ck_workspace_size": [p, i64, i64, i64, psz, psz],
        "ck_forward": [p, p, p, p, p, p, i64, i64, i64, p, p, sz, p, sz, p],
        "ck_backward": [p, p, p, i64, i64, i64, p, sz, p, p, p, p, p, p, p, sz, p],
        "ck_workspace_size_recompute": [p, i64, i64, i64, psz, psz],
        "ck_sgd_update": [p, p, i64, ctypes.c_float, p],
        "ck_adam_update": [p, p, p, p, i64, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                           ctypes.c_float, p, p],
        "ck_step_advance": [p, p],
        "ck_forward_checkpointed": [p, p, p, p, p, p, i64, i64, i64, p, p, sz, p, sz, p],
        "ck_backward_recompute": [p, p, p, p, p, i64, i64, i64, p, sz, p, p, p, p, p, p, p, sz, p],
        "ck_query_status": [p, p],
        "ck_query_status_static": [p],
        "ck_set_option": [ctypes.c_int, i64],
        "ck_forward_static_scratch": [p, p, p, p, p, p, i64, i64, i64, p, p, sz, p],
        "ck_probe_read": [p, sz, i64, p, p],
        "ck_probe_gather": [p, i64, i64, p, i64, p, p],
        "ck_probe_read_shape": [p, sz, i64, i64, i64, i64, i64, p, p],
        "ck_probe_grid_barrier": [i64, i64, i64, i64, i64, p, p, p, p],
        "ck_phase_profile_read": [p, i64, i64],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.ck_get_option.argtypes = [ctypes.c_int]
    lib.ck_get_option.restype = i64
    lib.ck_last_launch_count.argtypes = []
    lib.ck_last_launch_count.restype = i64
    lib.ck_status_string.argtypes = [ctypes.c_int]
    lib.ck_status_string.restype = ctypes.c_char_p
    lib.ck_last_error_message.argtypes = []
    lib.ck_last_error_message.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int):
    if status != CK_OK:
        raise CKError(status, load().ck_last_error_message().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def _shapes(handle, B: int, T: int, **tensors):
    """The library sees only pointers, so every tensor's shape is checked here
    against the graph's N, E, n_in and the call's B, T."""
    N, E, n_in = ck_graph_info(handle)
    want = {"edge_values": (E,), "d_edge_values": (E,), "leak": (N,), "d_leak": (N,),
            "bias": (N,), "d_bias": (N,), "drives": (T, n_in, B), "d_drives": (T, n_in, B),
            "state0": (B, N), "d_state0": (B, N), "states_out": (T, B, N), "d_states": (T, B, N)}
    for name, t in tensors.items():
        if t is None:
            if name in ("drives", "d_drives") and n_in == 0:
                continue
            raise ValueError(f"{name} is required")
        if tuple(t.shape) != want[name]:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {want[name]}")


def ck_graph_create(src, dst, num_nodes: int, input_nodes, stream=None, flags: int = 0):
    """ck_graph_create, or ck_graph_create_flags when flags is non-zero."""
    for t, n in ((src, "src"), (dst, "dst"), (input_nodes, "input_nodes")):
        _need(t, torch.int64, n)
    h = ctypes.c_void_p()
    n_in = 0 if input_nodes is None else input_nodes.numel()
    args = (_ptr(src), _ptr(dst), src.numel(), num_nodes, _ptr(input_nodes) if n_in else None, n_in)
    if flags:
        _check(load().ck_graph_create_flags(*args, int(flags), _stream(stream), ctypes.byref(h)))
    else:
        _check(load().ck_graph_create(*args, _stream(stream), ctypes.byref(h)))
    return h


def ck_graph_destroy(handle):
    _check(load().ck_graph_destroy(handle))


def ck_graph_info(handle):
    n, e, k = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(load().ck_graph_info(handle, ctypes.byref(n), ctypes.byref(e), ctypes.byref(k)))
    return n.value, e.value, k.value


def ck_graph_export(handle, device=None, stream=None):
    N, E, _ = ck_graph_info(handle)
    dev = device or torch.device("cuda", torch.cuda.current_device())
    mk = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    out = dict(row_ptr=mk(N + 1), col=mk(E), perm=mk(E), rowT_ptr=mk(N + 1), colT=mk(E),
               permT=mk(E), slot=mk(N))
    _check(load().ck_graph_export(handle, *(_ptr(out[k]) for k in
                                            ("row_ptr", "col", "perm", "rowT_ptr", "colT",
                                             "permT", "slot")), _stream(stream)))
    return out


def ck_workspace_size(handle, B: int, T: int, microsteps: int):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().ck_workspace_size(handle, B, T, microsteps, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def ck_forward(handle, edge_values, leak, bias, drives, state0, microsteps, states_out,
               saved, scratch, stream=None):
    for t, n in ((edge_values, "edge_values"), (leak, "leak"), (bias, "bias"),
                 (drives, "drives"), (state0, "state0"), (states_out, "states_out")):
        _need(t, torch.float32, n)
    B = state0.shape[0]
    T = states_out.shape[0]
    _shapes(handle, B, T, edge_values=edge_values, leak=leak, bias=bias, drives=drives,
            state0=state0, states_out=states_out)
    _check(load().ck_forward(handle, _ptr(edge_values), _ptr(leak), _ptr(bias),
                             _ptr(drives) if drives is not None and drives.numel() else None,
                             _ptr(state0), B, T, microsteps, _ptr(states_out),
                             _ptr(saved), saved.numel() * saved.element_size(),
                             _ptr(scratch), scratch.numel() * scratch.element_size(),
                             _stream(stream)))


def ck_backward(handle, edge_values, leak, B, T, microsteps, saved, d_states, d_edge_values,
                d_leak, d_bias, d_drives, d_state0, scratch, stream=None):
    for t, n in ((edge_values, "edge_values"), (leak, "leak"), (d_states, "d_states"),
                 (d_edge_values, "d_edge_values"), (d_leak, "d_leak"), (d_bias, "d_bias"),
                 (d_drives, "d_drives"), (d_state0, "d_state0")):
        _need(t, torch.float32, n)
    _shapes(handle, B, T, edge_values=edge_values, leak=leak, d_states=d_states,
            d_edge_values=d_edge_values, d_leak=d_leak, d_bias=d_bias, d_drives=d_drives,
            d_state0=d_state0)
    _check(load().ck_backward(handle, _ptr(edge_values), _ptr(leak), B, T, microsteps,
                              _ptr(saved), saved.numel() * saved.element_size(),
                              _ptr(d_states), _ptr(d_edge_values), _ptr(d_leak), _ptr(d_bias),
                              _ptr(d_drives) if d_drives is not None and d_drives.numel() else None,
                              _ptr(d_state0), _ptr(scratch),
                              scratch.numel() * scratch.element_size(), _stream(stream)))


def ck_sgd_update(param, grad, lr: float, stream=None):
    _need(param, torch.float32, "param")
    _need(grad, torch.float32, "grad")
    if param.shape != grad.shape:
        raise ValueError("param and grad differ in shape")
    _check(load().ck_sgd_update(_ptr(param), _ptr(grad), param.numel(), float(lr),
                                _stream(stream)))


def ck_adam_update(param, grad, m, v, step, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                   eps: float = 1e-8, stream=None):
    """Adam at the step number held by the device int64 tensor `step`."""
    for t, name in ((param, "param"), (grad, "grad"), (m, "m"), (v, "v")):
        _need(t, torch.float32, name)
        if t.shape != param.shape:
            raise ValueError(f"{name} differs in shape from param")
    _need(step, torch.int64, "step")
    _check(load().ck_adam_update(_ptr(param), _ptr(grad), _ptr(m), _ptr(v), param.numel(),
                                 float(lr), float(beta1), float(beta2), float(eps), _ptr(step),
                                 _stream(stream)))


def ck_step_advance(step, stream=None):
    _need(step, torch.int64, "step")
    _check(load().ck_step_advance(_ptr(step), _stream(stream)))


def ck_workspace_size_recompute(handle, B: int, T: int, microsteps: int):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().ck_workspace_size_recompute(handle, B, T, microsteps, ctypes.byref(a),
                                              ctypes.byref(b)))
    return a.value, b.value


def ck_forward_checkpointed(handle, edge_values, leak, bias, drives, state0, microsteps,
                            states_out, ckpt, scratch, stream=None):
    for t, n in ((edge_values, "edge_values"), (leak, "leak"), (bias, "bias"),
                 (drives, "drives"), (state0, "state0"), (states_out, "states_out")):
        _need(t, torch.float32, n)
    B = state0.shape[0]
    T = states_out.shape[0]
    _shapes(handle, B, T, edge_values=edge_values, leak=leak, bias=bias, drives=drives,
            state0=state0, states_out=states_out)
    _check(load().ck_forward_checkpointed(
        handle, _ptr(edge_values), _ptr(leak), _ptr(bias),
        _ptr(drives) if drives is not None and drives.numel() else None, _ptr(state0), B, T,
        microsteps, _ptr(states_out), _ptr(ckpt), ckpt.numel() * ckpt.element_size(),
        _ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream)))


def ck_backward_recompute(handle, edge_values, leak, bias, drives, B, T, microsteps, ckpt,
                          d_states, d_edge_values, d_leak, d_bias, d_drives, d_state0, scratch,
                          stream=None):
    for t, n in ((edge_values, "edge_values"), (leak, "leak"), (bias, "bias"),
                 (drives, "drives"), (d_states, "d_states"), (d_edge_values, "d_edge_values"),
                 (d_leak, "d_leak"), (d_bias, "d_bias"), (d_drives, "d_drives"),
                 (d_state0, "d_state0")):
        _need(t, torch.float32, n)
    _shapes(handle, B, T, edge_values=edge_values, leak=leak, bias=bias, drives=drives,
            d_states=d_states, d_edge_values=d_edge_values, d_leak=d_leak, d_bias=d_bias,
            d_drives=d_drives, d_state0=d_state0)
    has_in = drives is not None and drives.numel()
    _check(load().ck_backward_recompute(
        handle, _ptr(edge_values), _ptr(leak), _ptr(bias), _ptr(drives) if has_in else None, B, T,
        microsteps, _ptr(ckpt), ckpt.numel() * ckpt.element_size(), _ptr(d_states),
        _ptr(d_edge_values), _ptr(d_leak), _ptr(d_bias),
        _ptr(d_drives) if d_drives is not None and d_drives.numel() else None, _ptr(d_state0),
        _ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream)))


def ck_forward_static_scratch(handle, edge_values, leak, bias, drives, state0, microsteps,
                              states_out, saved, stream=None):
    for t, n in ((edge_values, "edge_values"), (leak, "leak"), (bias, "bias"),
                 (drives, "drives"), (state0, "state0"), (states_out, "states_out")):
        _need(t, torch.float32, n)
    B = state0.shape[0]
    T = states_out.shape[0]
    _shapes(handle, B, T, edge_values=edge_values, leak=leak, bias=bias, drives=drives,
            state0=state0, states_out=states_out)
    _check(load().ck_forward_static_scratch(
        handle, _ptr(edge_values), _ptr(leak), _ptr(bias),
        _ptr(drives) if drives is not None and drives.numel() else None, _ptr(state0), B, T,
        microsteps, _ptr(states_out), _ptr(saved), saved.numel() * saved.element_size(),
        _stream(stream)))


def ck_query_status(scratch, stream=None):
    _check(load().ck_query_status(_ptr(scratch), _stream(stream)))


def ck_graph_memory(handle):
    """(device bytes, pinned host bytes) the graph handle holds."""
    d, h = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load().ck_graph_memory(handle, ctypes.byref(d), ctypes.byref(h)))
    return d.value, h.value


TILING_KEYS = ("C", "G", "P", "max_rows", "max_fin", "max_chunk", "max_edges", "ptr_len")


def ck_graph_tiling(handle, direction: int) -> dict:
    """The shared-memory tiling of one direction (all zero when it has none)."""
    info = (ctypes.c_int64 * 8)()
    _check(load().ck_graph_tiling(handle, direction, info))
    return dict(zip(TILING_KEYS, list(info)))


def ck_graph_export_tiling(handle, direction: int, meta, ptr, col, perm, rowid, stream=None):
    _check(load().ck_graph_export_tiling(handle, direction, _ptr(meta), _ptr(ptr), _ptr(col),
                                         _ptr(perm), _ptr(rowid), _stream(stream)))


def ck_query_status_static(stream=None):
    _check(load().ck_query_status_static(_stream(stream)))


def ck_probe_read(buf, reps, sink, stream=None):
    _check(load().ck_probe_read(_ptr(buf), buf.numel() * buf.element_size(), reps, _ptr(sink),
                                _stream(stream)))


def ck_probe_read_shape(buf, reps, load_bytes, depth, threads, ctas_per_sm, sink, stream=None):
    _check(load().ck_probe_read_shape(_ptr(buf), buf.numel() * buf.element_size(), reps,
                                      load_bytes, depth, threads, ctas_per_sm, _ptr(sink),
                                      _stream(stream)))


def ck_probe_grid_barrier(scheme, ctas, cluster, crossings, rows_per_cta, rows, words, status,
                          stream=None):
    _need(words, torch.int32, "words")
    _need(status, torch.int32, "status")
    if words.numel() < PROBE_BARRIER_WORDS or status.numel() < 1:
        raise ValueError(f"words needs {PROBE_BARRIER_WORDS} elements, status one")
    if rows_per_cta > 0:
        _need(rows, torch.float32, "rows")
        if rows.numel() < ctas * rows_per_cta * 32:
            raise ValueError("rows holds fewer than ctas * rows_per_cta * 32 floats")
    _check(load().ck_probe_grid_barrier(scheme, ctas, cluster, crossings, rows_per_cta,
                                        _ptr(rows) if rows_per_cta > 0 else None, _ptr(words),
                                        _ptr(status), _stream(stream)))


def ck_phase_profile_read(clear: bool = True):
    """The profiling build's phase counters as nested lists
    [direction][CTA][word] of ints (layout in ck.h); raises CKError
    (CK_ERR_UNSUPPORTED) in every other build."""
    n = 2 * PHASE_PROFILE_CTAS * PHASE_PROFILE_WORDS
    buf = (ctypes.c_uint64 * n)()
    _check(load().ck_phase_profile_read(ctypes.cast(buf, ctypes.c_void_p), n, 1 if clear else 0))
    flat = list(buf)
    per = PHASE_PROFILE_CTAS * PHASE_PROFILE_WORDS
    return [[flat[d * per + c * PHASE_PROFILE_WORDS:d * per + (c + 1) * PHASE_PROFILE_WORDS]
             for c in range(PHASE_PROFILE_CTAS)] for d in range(2)]


def ck_probe_gather(rows, idx, sink, stream=None):
    _need(rows, torch.float32, "rows")
    _need(idx, torch.int32, "idx")
    _check(load().ck_probe_gather(_ptr(rows), rows.shape[0], rows.shape[1], _ptr(idx),
                                  idx.numel(), _ptr(sink), _stream(stream)))


def ck_set_option(opt: int, value: int):
    _check(load().ck_set_option(opt, int(value)))


def ck_get_option(opt: int) -> int:
    return int(load().ck_get_option(opt))


def ck_last_launch_count() -> int:
    return int(load().ck_last_launch_count())
