"""ctypes binding of the test library libfa_gb300_testing.so (include/fa_testing.h).

The test library holds device probes (exponentials, one-tile tcgen05 MMAs,
TMA and tensor-memory round trips, a bounded wait that must time out),
microbenchmarks and a host run of the work scheduler. It is built next to the
attention library by ``exact_attention_smem_gb300.build`` and is not part of
the attention library's ABI. Argument marshalling only.
"""
from __future__ import annotations

import ctypes
import os

import exact_attention_smem_gb300 as fa
from exact_attention_smem_gb300._lib import FA_OK, _ptr, _stream

TEST_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(fa.__file__)),
                             "libfa_gb300_testing.so")

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

SIGS = {
    "fa_test_last_error": (ctypes.c_char_p, []),
    "fa_test_get_device_error": (_I, [ctypes.POINTER(_I), _I]),
    "fa_test_exp2": (_I, [_P, _P, _I, _I, _P]),
    "fa_exp2_poly_host": (_F, [_F]),
    "fa_micro": (_I, [_I, _I, _P, _I, _P]),
    "fa_test_mma": (_I, [_P, _P, _P, _I, _I, _P]),
    "fa_test_mma_pair": (_I, [_P, _P, _P, _P, _I, _I, _P]),
    "fa_test_mma_fp8": (_I, [_P, _P, _P, _I, _I, _P]),
    "fa_test_roundtrip": (_I, [_P, _P, _P, _P]),
    "fa_test_wait_timeout": (_I, [_P, ctypes.c_double, _P]),
    "fa_sched_list": (_I, [_I, _I, _P, _I, _I, _I, _I, _I, _I, _I, _P, _I]),
}

_lib = None


def load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(TEST_LIB_PATH):
        raise RuntimeError(f"{TEST_LIB_PATH} is missing: build it with "
                           "`python -m exact_attention_smem_gb300.build`")
    lib = ctypes.CDLL(TEST_LIB_PATH)
    for name, (res, args) in SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status, where):
    if status != FA_OK:
        detail = load().fa_test_last_error().decode()
        raise RuntimeError(f"{where}: status {status}{': ' + detail if detail else ''}")


def fa_test_get_device_error(clear=True):
    code = ctypes.c_int(0)
    _check(load().fa_test_get_device_error(ctypes.byref(code), int(clear)),
           "fa_test_get_device_error")
    return code.value


def fa_test_exp2(x, y, mode, stream=None):
    _check(load().fa_test_exp2(_ptr(x), _ptr(y), x.numel(), mode, _stream(stream)), "fa_test_exp2")


def fa_micro(kind, iters, out_dev, ctas, stream=None):
    _check(load().fa_micro(kind, iters, _ptr(out_dev), ctas, _stream(stream)), "fa_micro")


def fa_exp2_poly_host(x: float) -> float:
    return float(load().fa_exp2_poly_host(x))


def fa_test_mma(A, B, C, mode, N, stream=None):
    _check(load().fa_test_mma(_ptr(A), _ptr(B), _ptr(C), mode, N, _stream(stream)), "fa_test_mma")


def fa_test_mma_pair(A, B, C, flags, mode, N, stream=None):
    _check(load().fa_test_mma_pair(_ptr(A), _ptr(B), _ptr(C), _ptr(flags), mode, N,
                                   _stream(stream)), "fa_test_mma_pair")


def fa_test_mma_fp8(A, B, C, mode, N, stream=None):
    _check(load().fa_test_mma_fp8(_ptr(A), _ptr(B), _ptr(C), mode, N, _stream(stream)),
           "fa_test_mma_fp8")


def fa_test_roundtrip(src, dst, tmem_out, stream=None):
    _check(load().fa_test_roundtrip(_ptr(src), _ptr(dst), _ptr(tmem_out), _stream(stream)),
           "fa_test_roundtrip")


def fa_test_wait_timeout(status_dev, timeout_ms, stream=None):
    _check(load().fa_test_wait_timeout(_ptr(status_dev), float(timeout_ms), _stream(stream)),
           "fa_test_wait_timeout")


def fa_sched_list(kind, B, cu_seqlens_host, Sq, Sk, heads, causal, grid, cta, heads_per_group=0):
    """Return the (seq, row block, head, cost) units of one CTA, in order."""
    lib = load()
    cu = None
    if cu_seqlens_host is not None:
        arr = (ctypes.c_int * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
        cu = ctypes.cast(arr, ctypes.c_void_p)
    n = lib.fa_sched_list(kind, B, cu, Sq, Sk, heads, int(causal), grid, cta, heads_per_group,
                          None, 0)
    if n < 0:
        raise ValueError("fa_sched_list: bad arguments")
    out = (ctypes.c_int * (4 * max(n, 1)))()
    lib.fa_sched_list(kind, B, cu, Sq, Sk, heads, int(causal), grid, cta, heads_per_group,
                      ctypes.cast(out, ctypes.c_void_p), n)
    return [tuple(out[4 * i:4 * i + 4]) for i in range(n)]
