"""Builds the CUDA library (libpa_gb300.so) in-tree with nvcc for sm_103a.

build(trace=True) builds the diagnostic variant libpa_gb300_trace.so instead:
the same sources compiled with PA_TRACE, whose kernels record the pipeline
timeline of pa_debug_set_trace (the default library carries no trace code).
build(debug=True) builds libpa_gb300_debug.so: the sources compiled with
PA_DEBUG (work-item bounds checks, shared and tensor memory poisoned before
first use).

Translation units compile in parallel, then link into one shared library next
to this file.  The seeded input generators (synth/csrc) are built the same way:
the device int8 generator into synth/libpa_synth.so (nvcc) and the threaded
host normal generator into synth/libpa_synth_host.so (gcc).  Rebuilds only when
a source is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libpa_gb300.so")
TRACE_LIB = os.path.join(PKG, "libpa_gb300_trace.so")
DEBUG_LIB = os.path.join(PKG, "libpa_gb300_debug.so")
SYNTH_SRC = os.path.join(ROOT, "synth", "csrc", "synth_gen.cu")
SYNTH_LIB = os.path.join(ROOT, "synth", "libpa_synth.so")
SYNTH_HOST_SRC = os.path.join(ROOT, "synth", "csrc", "synth_host.c")
SYNTH_HOST_LIB = os.path.join(ROOT, "synth", "libpa_synth_host.so")
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cuda, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(INCLUDE, "pa.h")]


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(verbose: bool = False, force: bool = False, trace: bool = False, debug: bool = False) -> str:
    if trace and debug:
        raise ValueError("the trace and debug libraries are separate builds")
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()
    deps = srcs + _headers()
    lib = TRACE_LIB if trace else DEBUG_LIB if debug else LIB
    if force or _stale(lib, deps):
        sub = os.path.join(BUILD_DIR, "trace") if trace else os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
        os.makedirs(sub, exist_ok=True)
        defs = ["-DPA_TRACE"] if trace else ["-DPA_DEBUG"] if debug else []
        objs = [os.path.join(sub, os.path.basename(s)[:-3] + ".o") for s in srcs]
        cmds = [[nvcc, *ARCH, *FLAGS, *defs, "-I", INCLUDE, "-I", CSRC, "-c", s, "-o", o]
                for s, o in zip(srcs, objs)]
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(cmds), os.cpu_count() or 4))) as ex:
            logs = list(ex.map(_run, cmds))
        if verbose:
            for lg in logs:
                print(lg)
        tmp = lib + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    if force or _stale(SYNTH_LIB, [SYNTH_SRC]):
        tmp = SYNTH_LIB + ".tmp"
        _run([nvcc, *ARCH, *FLAGS, "-shared", "-cudart", "shared", SYNTH_SRC, "-o", tmp])
        os.replace(tmp, SYNTH_LIB)
    if force or _stale(SYNTH_HOST_LIB, [SYNTH_HOST_SRC]):
        tmp = SYNTH_HOST_LIB + ".tmp"
        _run([shutil.which("gcc") or "gcc", "-O2", "-fPIC", "-shared", "-pthread", SYNTH_HOST_SRC,
              "-o", tmp, "-lm"])
        os.replace(tmp, SYNTH_HOST_LIB)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
