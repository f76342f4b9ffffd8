"""Build libzero.so in-tree for sm_103a (GB300).

Each translation unit under ``csrc/`` is compiled by nvcc in parallel, then
linked into ``zero_partitioned_mixed_replica_gb300/libzero.so`` with the CUDA
runtime linked statically.  ``python -m zero_partitioned_mixed_replica_gb300.build``
or :func:`build` from Python.  ``build(checked=True)`` (or ``--checked``)
builds the bounds-checked variant, ``libzero_checked.so``: the same sources
with -DZK_CHECKED, objects kept apart.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libzero.so")
OBJ_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libzero_checked.so")

SOURCES = ["zero_layout.cpp", "zero_rs.cu", "zero_adamw.cu", "zero_norm.cu", "zero_gather.cu",
           "zero_noalloc.cu", "zero_accum.cu", "zero_exec.cpp"]
HEADERS = ["zero_internal.h", "zero_device.cuh", "zero_launch.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no contraction of a*b+c on the device; the host compiler gets
# -ffp-contract=off for the same reason.
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-fmad=false",
                     "-Xcompiler", "-fPIC,-ffp-contract=off,-fno-strict-aliasing",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    obj_dir, lib = (OBJ_CHECKED, LIB_CHECKED) if checked else (OBJ, LIB)
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "zero.h")]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src + ".o")
        objs.append(o)
        if force or not _newer(o, [s] + hdrs):
            flags = list(NVCC_FLAGS) + (["-DZK_CHECKED"] if checked else [])
            if verbose_ptxas and src.endswith(".cu"):
                flags += ["-Xptxas", "-v"]
            jobs.append([nvcc, *flags, "-c", s, "-o", o])

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    failed = []
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for cmd, p in ex.map(run, jobs):
            if verbose_ptxas or p.returncode != 0:
                sys.stderr.write(p.stdout + p.stderr)
            if p.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or jobs or not _newer(lib, objs):
        tmp = lib + ".tmp%d" % os.getpid()
        subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv))
