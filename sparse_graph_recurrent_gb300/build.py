"""Build libck.so in-tree with nvcc for sm_103a (GB300).

Each .cu under csrc/ compiles to an object in parallel; the objects link into
sparse_graph_recurrent_gb300/_build/libck.so.  Rebuilds only when a source or
header is newer than the library.

Variant "bounds" builds the same sources with -DCK_DEBUG_BOUNDS into
_build/libck_bounds.so: every gathered row, table and carry index is checked
on the device, and a bad one is reported through ck_query_status instead of
being accessed.  The binding loads it when CK_LIBRARY_VARIANT=bounds.

Variant "prof" (-DCK_PHASE_PROFILE, _build/libck_prof.so) adds %globaltimer
stamps around each phase of a microstep, read with ck_phase_profile_read; the
binding loads it when CK_LIBRARY_VARIANT=prof.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libck.so")
VARIANTS = {None: ([], "libck.so"), "bounds": (["-DCK_DEBUG_BOUNDS"], "libck_bounds.so"),
            "prof": (["-DCK_PHASE_PROFILE"], "libck_prof.so")}


def lib_path(variant=None) -> str:
    if variant not in VARIANTS:
        raise ValueError(f"unknown library variant {variant!r}")
    return os.path.join(OUT, VARIANTS[variant][1])

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _inputs():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return srcs, deps


def build(force: bool = False, verbose: bool = False, variant=None) -> str:
    """Compile the library variant (None: the ordinary build) if a source is
    newer than it; return its path."""
    defines, name = VARIANTS[variant]
    lib = lib_path(variant)
    srcs, deps = _inputs()
    if not force and os.path.exists(lib):
        newest = max(os.path.getmtime(p) for p in deps)
        if os.path.getmtime(lib) >= newest:
            return lib
    objdir = os.path.join(OUT, "obj" if variant is None else "obj_" + variant)
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list:
    """Every variant, compiled side by side."""
    with ThreadPoolExecutor(max_workers=len(VARIANTS)) as ex:
        return list(ex.map(lambda v: build(force=force, variant=v), list(VARIANTS)))


if __name__ == "__main__":
    print(build(force=True, verbose=True))
