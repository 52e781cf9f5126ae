"""Builds libqdq.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel to an object file under ``_build/``;
the objects link into ``libqdq.so`` next to this file.  The CUDA runtime is
linked statically so the library only needs the NVIDIA driver at run time.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqdq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the qdq CUDA library cannot be built")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


LIB_CHECKED = os.path.join(PKG, "libqdq_checked.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checks")


def _stale(lib) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    deps.append(os.path.join(INCLUDE, "qdq.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, jobs: int | None = None, checks: bool = False) -> str:
    """Compile every kernel source and link libqdq.so; returns the library path.

    checks=True builds the debug variant libqdq_checked.so instead: the same sources with
    -DQDQ_CHECKS, whose kernels record out-of-bounds indices in a device status word
    (qdq_check_status) instead of accessing them.
    """
    bdir, lib = (BUILD_CHECKED, LIB_CHECKED) if checks else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(bdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DQDQ_CHECKS"] if checks else [])

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, os.cpu_count() or 4)) as ex:
        for err in ex.map(compile_one, zip(srcs, objs)):
            if verbose and err.strip():
                print(err)
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
