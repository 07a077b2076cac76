"""Build the C-ABI shared library ``libfa_gb300.so`` in-tree with nvcc (sm_103a).

Each ``csrc/*.cu`` is compiled in parallel to ``_build/*.o`` and linked with the
static CUDA runtime, so the library needs only the driver at run time (the
tensor-map encoder is reached through the runtime's driver entry point).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa_gb300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(PKG, "..", "include", "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, log):
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    if not _stale(obj, [src] + _headers()):
        return obj
    cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "a") as fh:
        fh.write(" ".join(cmd) + "\n" + r.stdout + r.stderr + "\n")
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
    return obj


def build(verbose: bool = False) -> str:
    """Compile and link the library if any source changed; return its path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    log = os.path.join(BUILD, "ptxas.log")
    if _stale(LIB, srcs + _headers()):
        if os.path.exists(log):
            os.remove(log)
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, log), srcs))
    if _stale(LIB, objs):
        # exported symbols: the extern "C" entry points (default visibility)
        cmd = [NVCC, *ARCH, "-shared", "-o", LIB + ".tmp", *objs, "-cudart", "static",
               "-Xlinker", "--exclude-libs,ALL", "-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(LIB + ".tmp", LIB)
    if verbose and os.path.exists(log):
        sys.stdout.write(open(log).read())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
