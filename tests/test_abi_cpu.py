"""Host-side checks of libck that need no GPU: it builds for sm_103a, loads,
exports every entry point include/ck.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_graph_recurrent_gb300 import _ck
    return _ck.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ck_[a-z_0-9]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"ck_graph_create", "ck_forward", "ck_backward", "ck_workspace_size"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


@pytest.mark.parametrize("variant", ["bounds", "prof"])
def test_every_build_exports_the_same_symbols(variant):
    """The bounds-checked (libck_bounds.so) and profiling (libck_prof.so)
    variants are the same ABI."""
    from sparse_graph_recurrent_gb300 import build
    lib_v = ctypes.CDLL(build.build(variant=variant))
    for n in sorted(_declared()):
        assert hasattr(lib_v, n), n


def test_phase_profile_only_in_the_profiling_build(lib):
    """The ordinary build keeps no phase profile and says so without touching
    the device (this runs without a GPU)."""
    lib.ck_phase_profile_read.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]
    buf = (ctypes.c_uint64 * 16)()
    assert lib.ck_phase_profile_read(ctypes.cast(buf, ctypes.c_void_p), 16, 1) == 7  # UNSUPPORTED
    assert b"profiling build" in lib.ck_last_error_message()


def test_status_strings(lib):
    for code, name in [(0, b"CK_OK"), (1, b"CK_ERR_INVALID_ARG"), (4, b"CK_ERR_TIMEOUT"),
                       (5, b"CK_ERR_WORKSPACE"), (7, b"CK_ERR_UNSUPPORTED")]:
        assert lib.ck_status_string(code) == name


def test_options_validate(lib):
    from sparse_graph_recurrent_gb300 import _ck
    assert _ck.ck_get_option(_ck.OPT_PERSISTENT) == 1
    assert _ck.ck_get_option(_ck.OPT_GRAPH_IN_SMEM) == 1
    with pytest.raises(_ck.CKError) as e:
        _ck.ck_set_option(_ck.OPT_BARRIER_TIMEOUT_NS, 10)
    assert e.value.name == "CK_ERR_INVALID_ARG"
    with pytest.raises(_ck.CKError) as e:
        _ck.ck_set_option(_ck.OPT_TEST_BARRIER_EXTRA, -1)
    assert e.value.name == "CK_ERR_INVALID_ARG"
    with pytest.raises(_ck.CKError) as e:
        _ck.ck_set_option(17, 1)
    assert e.value.name == "CK_ERR_INVALID_ARG"
    assert _ck.ck_get_option(_ck.OPT_BARRIER_TIMEOUT_NS) == 4_000_000_000
    # recompute window: default, round trip, range
    assert _ck.ck_get_option(_ck.OPT_RECOMPUTE_STEPS) == 0
    try:
        _ck.ck_set_option(_ck.OPT_RECOMPUTE_STEPS, 5)
        assert _ck.ck_get_option(_ck.OPT_RECOMPUTE_STEPS) == 5
        with pytest.raises(_ck.CKError) as e:
            _ck.ck_set_option(_ck.OPT_RECOMPUTE_STEPS, -1)
        assert e.value.name == "CK_ERR_INVALID_ARG"
        assert _ck.ck_get_option(_ck.OPT_RECOMPUTE_STEPS) == 5
    finally:
        _ck.ck_set_option(_ck.OPT_RECOMPUTE_STEPS, 0)


def test_graph_create_rejects_bad_sizes_before_cuda(lib):
    h = ctypes.c_void_p()
    # N < 1, negative E, n_in > N, NULL output: all refused on the host
    assert lib.ck_graph_create(None, None, 0, 0, None, 0, None, ctypes.byref(h)) == 1
    assert lib.ck_graph_create(None, None, -1, 4, None, 0, None, ctypes.byref(h)) == 1
    assert lib.ck_graph_create(None, None, 0, 4, None, 5, None, ctypes.byref(h)) == 1
    assert lib.ck_graph_create(None, None, 0, 4, None, 0, None, None) == 1
    assert lib.ck_graph_create(None, None, 3, 4, None, 0, None, ctypes.byref(h)) == 1  # NULL src
    assert b"NULL" in lib.ck_last_error_message()
    assert lib.ck_workspace_size(None, 1, 1, 1, None, None) == 1
    # graph flags: unknown bits refused before any CUDA call
    f = lib.ck_graph_create_flags
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    for bad in (4, 8, 1 << 31, 7):
        assert f(None, None, 0, 4, None, 0, bad, None, ctypes.byref(h)) == 1
        assert b"flag" in lib.ck_last_error_message()
    for ok in (1, 2, 3):  # valid flags: the call gets as far as the size check (N < 1)
        assert f(None, None, 0, 0, None, 0, ok, None, ctypes.byref(h)) == 1
        assert b"flag" not in lib.ck_last_error_message()


def test_no_cpu_fallback_without_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    src = (ctypes.c_int64 * 1)(0)
    st = lib.ck_graph_create(src, src, 1, 1, None, 0, None, ctypes.byref(h))
    assert st == 2 and not h.value  # CK_ERR_CUDA, no handle


def test_binding_constants_match_the_header():
    """The binding's option, scheme and size constants are the header's."""
    from sparse_graph_recurrent_gb300 import _ck
    text = open(os.path.join(ROOT, "include", "ck.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)

    def enum_values(prefix):
        vals = {}
        for name, val in re.findall(r"\b(" + prefix + r"[A-Z_0-9]+)\s*=\s*(\d+)", text):
            vals[name] = int(val)
        return vals

    schemes = enum_values("CK_BARRIER_")
    assert len(schemes) == 7
    for name, val in schemes.items():
        assert getattr(_ck, name[len("CK_"):]) == val, name
    opts = enum_values("CK_OPT_")
    for name, val in opts.items():
        assert getattr(_ck, "OPT_" + name[len("CK_OPT_"):]) == val, name
    words = re.search(r"#define\s+CK_PROBE_BARRIER_WORDS\s+(\d+)", text)
    assert words and int(words.group(1)) == _ck.PROBE_BARRIER_WORDS


def test_barrier_probe_refuses_bad_arguments_on_the_host(lib):
    """Argument checks come before any CUDA call (this runs without a GPU)."""
    assert lib.ck_probe_grid_barrier(9, 8, 1, 10, 0, None, None, None, None) == 1
    assert lib.ck_probe_grid_barrier(0, 8, 4, 10, 0, None, None, None, None) == 1
    assert b"scheme" in lib.ck_last_error_message()


def test_adam_refuses_bad_arguments_on_the_host(lib):
    """Argument checks of the Adam update come before any CUDA call."""
    f = lib.ck_adam_update
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] + [ctypes.c_float] * 4 + [ctypes.c_void_p] * 2
    one = (ctypes.c_int64 * 1)(1)
    step = ctypes.cast(one, ctypes.c_void_p)
    assert f(None, None, None, None, -1, 0.01, 0.9, 0.999, 1e-8, step, None) == 1   # n < 0
    assert f(None, None, None, None, 4, 0.01, 1.0, 0.999, 1e-8, step, None) == 1    # beta1 = 1
    assert f(None, None, None, None, 4, 0.01, 0.9, -0.1, 1e-8, step, None) == 1     # beta2 < 0
    assert f(None, None, None, None, 4, 0.01, 0.9, 0.999, 0.0, step, None) == 1     # eps = 0
    assert f(None, None, None, None, 4, float("nan"), 0.9, 0.999, 1e-8, step, None) == 1
    assert f(None, None, None, None, 4, 0.01, 0.9, 0.999, 1e-8, None, None) == 1    # no step
    assert f(None, None, None, None, 4, 0.01, 0.9, 0.999, 1e-8, step, None) == 1    # NULL arrays
    lib.ck_step_advance.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert lib.ck_step_advance(None, None) == 1
