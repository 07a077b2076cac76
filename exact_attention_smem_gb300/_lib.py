"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

Every function keeps the C name and argument order; tensors are passed as
torch tensors (their device pointers are handed to the library) and `stream`
as a torch.cuda.Stream or None (the current stream). No computation happens
here: the attention path runs entirely in the library's CUDA kernels, and the
library must be present — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

_lib = None

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ARCH = 3
FA_ERR_CUDA = 4
FA_ERR_WORKSPACE = 5
FA_ERR_TIMEOUT = 6

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

_SIGS = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P]),
    "fa_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                    ctypes.c_size_t, _P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                            _P, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                           _P, _P, _P, ctypes.c_size_t, _P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_last_error": (ctypes.c_char_p, []),
    "fa_get_device_error": (_I, [ctypes.POINTER(_I), _I]),
    "fa_debug_set": (_I, [ctypes.c_char_p, ctypes.c_double]),
    "fa_debug_set_events": (_I, [_I, _P, _P]),
    "fa_debug_set_trace": (_I, [_P, ctypes.c_size_t]),
    "fa_merge": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "fa_accumulate": (_I, [_P, _P, ctypes.c_longlong, _P]),
    "fa_to_bf16": (_I, [_P, _P, ctypes.c_longlong, _P]),
    "fa_quantize_fp8": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float,
                        _P]),
}


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.fa_status_string(status).decode()
        detail = lib.fa_last_error().decode()
        super().__init__(f"{where}: {msg} ({status}){': ' + detail if detail else ''}")
        self.status = status


def load():
    """Load the library (built by exact_attention_smem_gb300.build); raise if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m exact_attention_smem_gb300.build` "
            "(the attention path has no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    return list(_SIGS)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != FA_OK:
        raise FAError(status, where)


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, cu_seqlens=None, stream=None):
    _check(load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, d,
                         int(causal), float(scale), _ptr(cu_seqlens), _stream(stream)), "fa_fwd")


def fa_fwd_varlen(q, k, v, o, lse, nseq, Hq, Hkv, Tq, Tk, d, causal, scale, cu_q, cu_k,
                  stream=None):
    _check(load().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), nseq, Hq, Hkv, Tq,
                                Tk, d, int(causal), float(scale), _ptr(cu_q), _ptr(cu_k),
                                _stream(stream)), "fa_fwd_varlen")


def fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, nseq, Hq, Hkv, Tq, Tk, d, causal, scale,
                  cu_q, cu_k, workspace, workspace_bytes, stream=None):
    _check(load().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                _ptr(dq), _ptr(dk), _ptr(dv), nseq, Hq, Hkv, Tq, Tk, d,
                                int(causal), float(scale), _ptr(cu_q), _ptr(cu_k),
                                _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "fa_bwd_varlen")


def fa_bwd_workspace_bytes(B, Hq, Sq, d, total_q=0):
    return int(load().fa_bwd_workspace_bytes(B, Hq, Sq, d, total_q))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
           cu_seqlens, workspace, workspace_bytes, stream=None):
    _check(load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, d, int(causal), float(scale),
                         _ptr(cu_seqlens), _ptr(workspace), int(workspace_bytes),
                         _stream(stream)), "fa_bwd")


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
                   cu_seqlens=None, stream=None):
    """fa_bwd with the library's built-in scratch instead of a caller workspace."""
    _check(load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, d, int(causal),
                                 float(scale), _ptr(cu_seqlens), _stream(stream)),
           "fa_bwd_noalloc")


def fa_get_device_error(clear=True):
    code = ctypes.c_int(0)
    _check(load().fa_get_device_error(ctypes.byref(code), int(clear)), "fa_get_device_error")
    return code.value


def fa_debug_set(key, value):
    _check(load().fa_debug_set(key.encode(), float(value)), "fa_debug_set")


def fa_debug_set_events(which, start=None, stop=None):
    """Arm one-shot timing events (torch.cuda.Event) around the next fwd/bwd main kernel."""
    def h(ev):
        if ev is None:
            return None
        if not ev.cuda_event:
            ev.record()          # torch creates the CUDA event lazily
            ev.synchronize()
        return ctypes.c_void_p(ev.cuda_event)
    _check(load().fa_debug_set_events(which, h(start), h(stop)), "fa_debug_set_events")


def fa_debug_set_trace(buf=None):
    """Arm (device int64 tensor) or disarm (None) the backward role timeline."""
    _check(load().fa_debug_set_trace(_ptr(buf), 0 if buf is None else buf.numel() * 8),
           "fa_debug_set_trace")


def fa_merge(o_parts, lse_parts, P, B, Hq, S, d, packed, o, lse, stream=None):
    _check(load().fa_merge(_ptr(o_parts), _ptr(lse_parts), P, B, Hq, S, d, int(packed), _ptr(o),
                           _ptr(lse), _stream(stream)), "fa_merge")


def fa_quantize_fp8(x, B, S, H, d, layout, codes, scales, stream=None):
    _check(load().fa_quantize_fp8(_ptr(x), B, S, H, d, layout, _ptr(codes), _ptr(scales),
                                  _stream(stream)), "fa_quantize_fp8")


def fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, B, Hq, Hkv, Sq, Sk, d, causal,
               scale, stream=None):
    _check(load().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(q_scale), _ptr(k_scale),
                             _ptr(v_scale), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, d,
                             int(causal), float(scale), _stream(stream)), "fa_fwd_fp8")


def fa_accumulate(acc, x, n=None, stream=None):
    """acc (fp32) += x (bf16), element-wise over n elements (default: all of x)."""
    n = x.numel() if n is None else n
    _check(load().fa_accumulate(_ptr(acc), _ptr(x), int(n), _stream(stream)), "fa_accumulate")


def fa_to_bf16(out, x, n=None, stream=None):
    """out (bf16) = x (fp32) rounded to nearest even, over n elements (default: all of x)."""
    n = x.numel() if n is None else n
    _check(load().fa_to_bf16(_ptr(out), _ptr(x), int(n), _stream(stream)), "fa_to_bf16")
