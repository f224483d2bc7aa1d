"""Builds libgdn.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a only.

Each ``csrc/*.cu`` file is compiled to an object in ``_build/`` in parallel, then linked into
``libgdn.so`` next to this file.  The same sources are compiled a second time with
``-DGDN_TEST_HOOKS`` into ``_build/test/`` and linked into ``libgdn_test.so``: the verification
hooks of ``include/gdn_debug.h`` (chunk-design selection, a one-tile MMA check, a dropped copy
that makes a bounded wait run out) exist only there, so the product library carries no switch that
changes results and no fault hook.  Objects are rebuilt when their source or any shared header is
newer.  Usage: ``python -m linear_attention_ssm_gb300.build`` or ``build()`` from Python.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgdn.so")
TEST_LIB = os.path.join(HERE, "libgdn_test.so")
# sources that only the test library holds
TEST_ONLY = ("debug_probe.cu",)
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", INCLUDE, "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn.so")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _build_lib(lib, objdir, sources, flags, cc, headers, verbose):
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        if _stale(obj, [src] + headers):
            cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr, flush=True)
        return obj
    return compile_one


def _link(lib, objs, cc):
    if _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)


def build(verbose: bool = False, extra_flags=None, test_library: bool = True) -> str:
    """Compile and link libgdn.so (and, unless test_library is False, libgdn_test.so); returns
    the product library's path."""
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    product = [s for s in sources if os.path.basename(s) not in TEST_ONLY]
    headers = _headers()
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])
    jobs = [(LIB, BUILD, product, flags)]
    if test_library:
        jobs.append((TEST_LIB, os.path.join(BUILD, "test"), sources, flags + ["-DGDN_TEST_HOOKS=1"]))
    work = []
    for lib, objdir, srcs, fl in jobs:
        fn = _build_lib(lib, objdir, srcs, fl, cc, headers, verbose)
        work += [(fn, s) for s in srcs]
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4, len(work))) as ex:
        objs = list(ex.map(lambda w: w[0](w[1]), work))
    i = 0
    for lib, objdir, srcs, fl in jobs:
        _link(lib, objs[i:i + len(srcs)], cc)
        i += len(srcs)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
