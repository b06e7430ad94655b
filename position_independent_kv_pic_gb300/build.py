"""Build the C-ABI library libpic.so in-tree for sm_103a (GB300).

Every .cu under csrc/ is compiled by nvcc for ``-gencode arch=compute_103a,code=sm_103a``
and the host-only .cpp files by g++, in parallel; the objects are linked into
``position_independent_kv_pic_gb300/libpic.so`` with the CUDA runtime linked statically,
so the library loads on a machine without a GPU driver (its symbols can be inspected
there) and needs only the driver on a GPU machine.

Usage: ``python -m position_independent_kv_pic_gb300.build [--force]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found")
    return p


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu"))), sorted(glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _up_to_date(lib: str) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False, extra_nvcc=(), name: str = "libpic.so") -> str:
    """Compile and link the library; returns its path.  Skips work when up to date.

    ``name`` other than libpic.so builds a variant of the library (its own objects
    and file, next to libpic.so) with ``extra_nvcc`` added, e.g. the failure-injection
    test build; a variant is rebuilt only when it is missing or older than a source."""
    lib = os.path.join(PKG, name)
    variant = name != "libpic.so"
    if not force and (variant or not extra_nvcc) and _up_to_date(lib):
        return lib
    bdir = os.path.join(BUILD, os.path.splitext(name)[0]) if variant else BUILD
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    cus, cpps = _sources()
    jobs = []
    for src in cus:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        jobs.append(([nvcc, *ARCH, *NVCC_FLAGS, *extra_nvcc, "-c", src, "-o", obj], obj))
    for src in cpps:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        jobs.append((["g++", *CXX_FLAGS, "-c", src, "-o", obj], obj))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        outs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose:
        for o in outs:
            if o.strip():
                print(o)
    tmp = lib + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for _, o in jobs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    force = "--force" in sys.argv
    verbose = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force=force or bool(extra), verbose=verbose or bool(extra), extra_nvcc=extra))
