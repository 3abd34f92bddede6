"""In-tree build of libpurlin.so (the C-ABI CUDA library) for sm_103a.

Every translation unit is compiled by nvcc in parallel, then linked into
``reduce_datapath_gb300/lib/libpurlin.so``.  No cmake, no setuptools: one
``-gencode`` (compute_103a / sm_103a), ``-lineinfo`` for profiling, no fast-math.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libpurlin.so")

SOURCES = ["capi.cpp", "layout.cpp", "zs_kernels.cu", "snac_kernels.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-Xcompiler", "-fvisibility=hidden",
          "-I", INCLUDE, "-I", CSRC]
CUDA_ONLY = ARCH + ["-lineinfo", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.exists(os.path.join(home, "bin", "nvcc")):
        return os.path.join(home, "bin", "nvcc")
    found = shutil.which("nvcc")
    if found:
        return found
    if os.path.exists("/usr/local/cuda/bin/nvcc"):
        return "/usr/local/cuda/bin/nvcc"
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


# The checked build: the same sources with PURLIN_CHECKED (every kernel access
# tested against the call's buffers), for tests.
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(LIBDIR, "libpurlin_checked.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def is_fresh(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile_jobs(build_dir: str, defines: list, verbose: bool):
    """Start one nvcc per translation unit; returns [(src, obj, process)]."""
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    jobs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.rsplit(".", 1)[0] + ".o")
        cmd = [cc, *COMMON, *defines]
        if src.endswith(".cu"):
            cmd += CUDA_ONLY
        cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        jobs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    return jobs


def _finish(jobs, lib: str, verbose: bool) -> None:
    failed = []
    for src, _, p in jobs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"--- {src}\n{out}")
        elif verbose and out.strip():
            print(out, file=sys.stderr)
    if failed:
        raise RuntimeError(f"{os.path.basename(lib)} build failed:\n" + "\n".join(failed))
    tmp = lib + ".%d.tmp" % os.getpid()
    link = [nvcc(), "-shared", *ARCH, "-o", tmp, *[obj for _, obj, _ in jobs]]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"{os.path.basename(lib)} link failed:\n" + r.stdout)
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link libpurlin.so (checked=True: libpurlin_checked.so)
    unless it is newer than every source."""
    lib = LIB_CHECKED if checked else LIB
    if not force and is_fresh(lib):
        return lib
    os.makedirs(LIBDIR, exist_ok=True)
    jobs = _compile_jobs(BUILD_CHECKED if checked else BUILD,
                         ["-DPURLIN_CHECKED"] if checked else [], verbose)
    _finish(jobs, lib, verbose)
    return lib


def build_all(force: bool = False, verbose: bool = False) -> None:
    """Both libraries, every translation unit compiled at once."""
    os.makedirs(LIBDIR, exist_ok=True)
    pending = []
    for lib, d, defs in ((LIB, BUILD, []), (LIB_CHECKED, BUILD_CHECKED, ["-DPURLIN_CHECKED"])):
        if force or not is_fresh(lib):
            pending.append((lib, _compile_jobs(d, defs, verbose)))
    for lib, jobs in pending:
        _finish(jobs, lib, verbose)


if __name__ == "__main__":
    build_all(force="--force" in sys.argv, verbose=True)
    print(LIB, LIB_CHECKED)
