"""Build libtfqmm.so in-tree with nvcc for sm_103a (one -gencode, parallel units).

Two libraries come out of the same sources: libtfqmm.so (the product) and
libtfqmm_debug.so, built with TF_DEBUG_BOUNDS, whose kernels check every shared-
and global-memory index against its buffer and report a violation through the
device status word (TF_EBOUNDS) instead of making the access.  build_trace()
makes a third on request, libtfqmm_trace.so (TF_TRACE): per-CTA phase times of
every row-kernel launch (include/tfqmm_trace.h).
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
SO = os.path.join(OUT, "libtfqmm.so")
SO_DEBUG = os.path.join(OUT, "libtfqmm_debug.so")
SO_TRACE = os.path.join(OUT, "libtfqmm_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
VARIANTS = ((SO, OUT, []), (SO_DEBUG, os.path.join(OUT, "debug"), ["-DTF_DEBUG_BOUNDS"]))
TRACE_VARIANT = (SO_TRACE, os.path.join(OUT, "trace"), ["-DTF_TRACE"])


def _nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """The product and the bounds-checking libraries; returns the product's path."""
    _build(VARIANTS, force, verbose)
    return SO


def build_trace(force: bool = False, verbose: bool = False) -> str:
    """The phase-trace library; returns its path."""
    _build((TRACE_VARIANT,), force, verbose)
    return SO_TRACE


def _build(variants, force: bool, verbose: bool) -> None:
    nvcc = _nvcc()
    units = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    jobs = []
    for (_, out, defs) in variants:
        os.makedirs(out, exist_ok=True)
        for src in units:
            jobs.append((src, os.path.join(out, os.path.basename(src)[:-3] + ".o"), defs))

    def compile_unit(job) -> str:
        src, obj, defs = job
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, *FLAGS, *defs, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd))
            subprocess.check_call(cmd)
        return obj

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_unit, jobs))
    for i, (so, _, _) in enumerate(variants):
        mine = objs[i * len(units):(i + 1) * len(units)]
        if force or _stale(so, mine):
            tmp = so + ".tmp%d" % os.getpid()
            # -Bsymbolic: each library binds its own symbols first (both may share a process).
            subprocess.check_call([nvcc, *ARCH, "-shared", "-Xlinker", "-Bsymbolic", "-o", tmp, *mine])
            os.replace(tmp, so)


if __name__ == "__main__":
    print(build(verbose=True))
