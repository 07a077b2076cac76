"""Build the C-ABI shared libraries in-tree with nvcc (sm_103a).

``libfa_gb300.so`` (include/fa.h) is the attention library: every
``csrc/*.cu``. ``libfa_gb300_testing.so`` (include/fa_testing.h) holds the
probes and microbenchmarks the tests use (``csrc/testing/*.cu`` plus the shared
host helpers); the attention library does not contain them. Sources are
compiled in parallel to ``_build/`` and linked with the static CUDA runtime, so
each library needs only the driver at run time (the tensor-map encoder is
reached through the runtime's driver entry point).
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
TEST_LIB = os.path.join(PKG, "libfa_gb300_testing.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _test_sources():
    return sorted(glob.glob(os.path.join(CSRC, "testing", "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(PKG, "..", "include", "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, log):
    sub = "testing_" if os.path.basename(os.path.dirname(src)) == "testing" else ""
    obj = os.path.join(BUILD, sub + os.path.basename(src)[:-3] + ".o")
    if not _stale(obj, [src] + _headers()):
        return obj
    cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "a") as fh:
        fh.write(" ".join(cmd) + "\n" + r.stdout + r.stderr + "\n")
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
    return obj


def _link(lib, objs):
    if not _stale(lib, objs):
        return
    # exported symbols: the extern "C" entry points (default visibility)
    cmd = [NVCC, *ARCH, "-shared", "-o", lib + ".tmp", *objs, "-cudart", "static",
           "-Xlinker", "--exclude-libs,ALL", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed for {os.path.basename(lib)}:\n{r.stderr[-4000:]}")
    os.replace(lib + ".tmp", lib)


def build(verbose: bool = False) -> str:
    """Compile and link both libraries if any source changed; return the attention
    library's path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs, tsrcs = _sources(), _test_sources()
    log = os.path.join(BUILD, "ptxas.log")
    if _stale(LIB, srcs + _headers()) or _stale(TEST_LIB, tsrcs + _headers()):
        if os.path.exists(log):
            os.remove(log)
    with ThreadPoolExecutor(max_workers=min(8, len(srcs) + len(tsrcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, log), srcs + tsrcs))
    lib_objs, test_objs = objs[:len(srcs)], objs[len(srcs):]
    _link(LIB, lib_objs)
    common = [o for o in lib_objs if os.path.basename(o) == "host_common.o"]
    _link(TEST_LIB, test_objs + common)
    if verbose and os.path.exists(log):
        sys.stdout.write(open(log).read())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
