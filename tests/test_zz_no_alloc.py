"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Runtimes whose device memory is entirely managed by their own pool allocator,
or latency-critical paths where cudaMalloc (which may synchronise the device)
is off limits, cannot hand fa_bwd a workspace. fa_bwd_noalloc uses a fixed
scratch array inside the library instead. This file is named to be collected
last: it checks, through the C ABI, that two calls in a row give the same
gradients as fa_bwd with a caller workspace (within the gradient tolerance the
other tests use), and that a problem larger than the built-in scratch is
rejected before any work.
"""
import ctypes

import pytest
import torch

import exact_attention_smem_gb300 as fa
from attn_inputs import random_inputs
from exact_attention_smem_gb300 import _lib
from gpu_helpers import GRAD_TOL

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


def _dims(x):
    B, Sq, Hq, d = x.q.shape
    return B, Hq, x.k.shape[2], Sq, x.k.shape[1], d


def _rel(a, b):
    a, b = a.float(), b.float()
    return ((a - b).norm() / b.norm().clamp_min(1e-30)).item()


def test_noalloc_backward_matches_workspace_backward_twice():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    x = random_inputs(B=2, Hq=4, Hkv=2, Sq=700, Sk=700, d=128, seed=91, device="cuda")
    B, Hq, Hkv, Sq, Sk, d = _dims(x)
    scale = d ** -0.5
    assert fa.fa_bwd_workspace_bytes(B, Hq, Sq, d, 0) <= SCRATCH_BYTES
    o, lse = fa.forward(x.q, x.k, x.v, causal=True, scale=scale)
    ref = fa.backward(x.q, x.k, x.v, o, lse, x.do, causal=True, scale=scale)
    lib = _lib.load()
    for _ in range(2):
        dq, dk, dv = torch.empty_like(x.q), torch.empty_like(x.k), torch.empty_like(x.v)
        status = lib.fa_bwd_noalloc(
            _lib._ptr(x.q), _lib._ptr(x.k), _lib._ptr(x.v), _lib._ptr(o), _lib._ptr(lse),
            _lib._ptr(x.do), _lib._ptr(dq), _lib._ptr(dk), _lib._ptr(dv), B, Hq, Hkv, Sq, Sk, d,
            1, scale, None, _lib._stream(None))
        assert status == 0, lib.fa_last_error()
        torch.cuda.synchronize()
        assert fa.fa_get_device_error(clear=True) == 0
        for got, want in zip((dq, dk, dv), ref):
            assert torch.isfinite(got.float()).all()
            assert _rel(got, want) <= GRAD_TOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    fa.load()
    lib = _lib.load()
    B, Hq, S, d = 1, 32, 4096, 128           # needs > 32 MiB of scratch
    assert fa.fa_bwd_workspace_bytes(B, Hq, S, d, 0) > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x7F0000000000)  # rejected before any pointer is used
    status = lib.fa_bwd_noalloc(*([fake] * 9), B, Hq, Hq, S, S, d, 1, 0.1, None, None)
    assert status == 5
    assert b"scratch" in lib.fa_last_error()
