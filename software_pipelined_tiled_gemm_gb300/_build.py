"""Build the CUDA library libspgemm.so in-tree with nvcc (sm_103a only).

Each .cu file is compiled in parallel to an object under ``_build/`` and the
objects are linked into ``_lib/libspgemm.so`` (CUDA runtime linked
statically, so the library loads on a machine without a GPU driver; the
driver is reached at run time through the runtime's entry-point query).
A stamp of the sources' content hash decides whether a rebuild is needed.

The bounds-checked build (``checked=True``) compiles the same sources with
``-DSPGEMM_BOUNDS_CHECKS=1`` into ``_build_checked/`` and
``_lib/libspgemm_checked.so``: its kernels range-check the indexes and copy
coordinates they derive and report a failed check as GEMM_ERR_BOUNDS.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libspgemm.so")
STAMP = os.path.join(LIBDIR, "libspgemm.stamp")
LIB_CHECKED = os.path.join(LIBDIR, "libspgemm_checked.so")
STAMP_CHECKED = os.path.join(LIBDIR, "libspgemm_checked.stamp")
CHECKED_FLAGS = ["-DSPGEMM_BOUNDS_CHECKS=1"]

SOURCES = ["gemm_api.cu", "gemm_bn64.cu", "gemm_bn128.cu", "gemm_bn256.cu", "gemm_pair128.cu",
           "gemm_pair256.cu", "pad.cu", "fill.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspgemm.so")


def _digest(checked: bool = False) -> str:
    h = hashlib.sha256()
    files = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h")))
    for f in files:
        h.update(f.encode())
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(INCLUDE, "gemm.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS + (CHECKED_FLAGS if checked else [])).encode())
    return h.hexdigest()


KERNEL_FILES = ["gemm_kernel.cuh", "epilogue_math.cuh", "ptx.cuh", "kernel_params.h",
                "byte_shift.cuh", "gemm_instance.cuh",
                "gemm_bn64.cu", "gemm_bn128.cu", "gemm_bn256.cu", "gemm_pair128.cu",
                "gemm_pair256.cu"]


def _code_only(text: str) -> str:
    """C/C++ source with comments removed and each line stripped of
    surrounding whitespace (blank lines dropped); string and character
    literals are kept as they are."""
    out = []
    i, n = 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.strip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def _portable_flags() -> str:
    """The compiler flags with the include directories named relative to the
    repository, so that a checkout in another directory hashes the same."""
    rel = {CSRC: "software_pipelined_tiled_gemm_gb300/csrc", INCLUDE: "include"}
    return " ".join(ARCH + [rel.get(f, f) for f in FLAGS])


def kernel_digest() -> str:
    """Hash of the GEMM kernel's device code only (what an ncu capture of the
    kernel depends on): comments and layout do not count, the host planner is
    left out, and so is the directory the repository sits in."""
    h = hashlib.sha256()
    for f in KERNEL_FILES:
        h.update(f.encode())
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    h.update(_portable_flags().encode())
    return h.hexdigest()[:16]


def _paths(checked: bool):
    return (BUILD_CHECKED, LIB_CHECKED, STAMP_CHECKED) if checked else (BUILD, LIB, STAMP)


def up_to_date(checked: bool = False) -> bool:
    _, lib, stamp = _paths(checked)
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return False
    with open(stamp) as f:
        return f.read().strip() == _digest(checked)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link the library (or its bounds-checked build) if its
    sources changed; return its path."""
    return build_many([checked], force=force, verbose=verbose)[0]


def build_many(variants, force: bool = False, verbose: bool = False):
    """Build several variants (False: normal, True: bounds-checked), all their
    translation units compiled in one parallel pool; return their paths."""
    todo = [c for c in variants if force or not up_to_date(c)]
    if todo:
        nvcc = _nvcc()
        os.makedirs(LIBDIR, exist_ok=True)
        for c in todo:
            os.makedirs(_paths(c)[0], exist_ok=True)

        def compile_one(job):
            checked, src = job
            obj = os.path.join(_paths(checked)[0], src.replace(".cu", ".o"))
            cmd = ([nvcc] + ARCH + FLAGS + (CHECKED_FLAGS if checked else [])
                   + ["-c", os.path.join(CSRC, src), "-o", obj])
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
            return obj

        jobs = [(c, src) for c in todo for src in SOURCES]
        workers = max(1, min(len(jobs), os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
            objs = list(ex.map(compile_one, jobs))
        for c in todo:
            _, lib, stamp = _paths(c)
            mine = [o for (cc, _), o in zip(jobs, objs) if cc == c]
            tmp = lib + ".tmp%d" % os.getpid()
            cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + mine + ["-cudart", "static", "-ldl"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
            os.replace(tmp, lib)
            with open(stamp, "w") as f:
                f.write(_digest(c))
    return [_paths(c)[1] for c in variants]


if __name__ == "__main__":
    print(build_many([False, True], force=True, verbose=True))
