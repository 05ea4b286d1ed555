"""Builds the CUDA library ``_lib/libmoe.so`` in-tree, for sm_103a only.

Each ``csrc/*.cu`` file is compiled by its own nvcc process (in parallel) and
the objects are linked into one shared library with the CUDA runtime linked
statically.  The library exports only the C ABI of ``include/moe.h``.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_lib")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(OUT, "libmoe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                 "-I", INCLUDE, "-I", SRC, "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources():
    return sorted(os.path.join(SRC, f) for f in os.listdir(SRC) if f.endswith(".cu"))


def _deps():
    files = _sources() + [os.path.join(SRC, f) for f in os.listdir(SRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "moe.h"))
    return files


# Library variants: the normal one, and "bounds", compiled with MOE_DEBUG_BOUNDS
# (device-side checks of layout-derived indices, reported as MOE_DEVERR_BOUNDS;
# a debugging aid, not the product path).
VARIANTS = {"": ("libmoe.so", OUT, ()), "bounds": ("libmoe_bounds.so", os.path.join(OUT, "bounds"),
                                                   ("-DMOE_DEBUG_BOUNDS",))}


def library_path(variant: str = "") -> str:
    name, _, _ = VARIANTS[variant]
    return os.path.join(OUT, name)


def up_to_date(variant: str = "") -> bool:
    lib = library_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    """Compile (if needed) and return the path of the library (libmoe.so, or
    with variant="bounds" the bounds-checked libmoe_bounds.so)."""
    lib_path = library_path(variant)
    _, obj_dir, variant_flags = VARIANTS[variant]
    if not force and up_to_date(variant):
        return lib_path
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for src in _sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        jobs.append((src, obj, [nvcc, *CFLAGS, *variant_flags, *extra_flags, "-c", src, "-o", obj]))

    def run(job):
        src, obj, cmd = job
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{p.stdout}\n{p.stderr}")
        return p.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        logs = list(ex.map(run, jobs))
    if verbose:
        for log in logs:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[j[1] for j in jobs], "-cudart", "static"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
