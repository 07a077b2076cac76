"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Runtimes whose device memory is entirely managed by their own pool allocator,
or latency-critical paths where cudaMalloc (which may synchronise the device)
is off limits, cannot hand fa_bwd a workspace. fa_bwd_noalloc uses a fixed
scratch array inside the library instead. This file is named to be collected
last. Through the C ABI it checks that:

* two calls in a row give exactly the gradients of fa_bwd with a caller
  workspace (the default two-pass backward is bitwise reproducible), for a
  dense and a packed batch, and that they match the fp64 oracle;
* the one-pass form (fp32 dQ accumulator in the shared scratch, which the
  first call leaves non-zero) gives the right gradients on the second call
  too (within the gradient tolerance: its dQ uses atomics);
* a problem larger than the built-in scratch is rejected before any work.
"""
import ctypes
import os
import re

import pytest
import torch

import exact_attention_smem_gb300 as fa
import oracle
from attn_inputs import random_inputs
from exact_attention_smem_gb300 import _lib
from gpu_helpers import GRAD_TOL, rel_l2

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _scratch_bytes():
    """FA_BWD_NOALLOC_SCRATCH_BYTES as include/fa.h defines it."""
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    m = re.search(r"#define\s+FA_BWD_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "FA_BWD_NOALLOC_SCRATCH_BYTES not found in fa.h"
    return int(m.group(1)) << int(m.group(2))


@pytest.fixture(autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    yield
    fa.fa_debug_set("bwd_mode", 1)


def _noalloc(q, k, v, o, lse, do, B, Hq, Hkv, Sq, Sk, d, causal, scale, cu):
    lib = _lib.load()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    status = lib.fa_bwd_noalloc(
        _lib._ptr(q), _lib._ptr(k), _lib._ptr(v), _lib._ptr(o), _lib._ptr(lse), _lib._ptr(do),
        _lib._ptr(dq), _lib._ptr(dk), _lib._ptr(dv), B, Hq, Hkv, Sq, Sk, d, int(causal), scale,
        _lib._ptr(cu), _lib._stream(None))
    assert status == 0, lib.fa_last_error()
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    return dq, dk, dv


def _cases():
    x = random_inputs(B=2, Hq=4, Hkv=2, Sq=700, Sk=700, d=128, seed=91, device="cuda")
    yield "dense", (x.q, x.k, x.v, x.do, None), (2, 4, 2, 700, 700, 128)
    lengths = [300, 1, 0, 517, 129]
    x = random_inputs(B=None, Hq=4, Hkv=2, Sq=None, Sk=None, d=128, seed=92, lengths=lengths,
                      device="cuda")
    T = sum(lengths)
    yield "packed", (x.q, x.k, x.v, x.do, x.cu_seqlens), (len(lengths), 4, 2, T, T, 128)


def test_noalloc_backward_equals_workspace_backward_twice():
    limit = _scratch_bytes()
    for name, (q, k, v, do, cu), (B, Hq, Hkv, Sq, Sk, d) in _cases():
        scale = d ** -0.5
        assert fa.fa_bwd_workspace_bytes(B, Hq, Sq, d, Sq if cu is not None else 0) <= limit
        o, lse = fa.forward(q, k, v, causal=True, scale=scale, cu_seqlens=cu)
        ref = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, cu_seqlens=cu)
        torch.cuda.synchronize()
        exact = oracle.backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, True,
                                cu_seqlens=None if cu is None else cu.cpu())
        for _ in range(2):
            got = _noalloc(q, k, v, o, lse, do, B, Hq, Hkv, Sq, Sk, d, True, scale, cu)
            for g, want, ex in zip(got, ref, exact):
                assert torch.equal(g, want), name
                assert rel_l2(g, ex) <= GRAD_TOL, name


def test_noalloc_one_pass_form_starts_from_a_cleared_accumulator():
    """The one-pass form keeps an fp32 dQ accumulator in the shared scratch;
    the second call must not add onto what the first call left there."""
    fa.fa_debug_set("bwd_mode", 0)
    x = random_inputs(B=1, Hq=4, Hkv=4, Sq=513, Sk=513, d=128, seed=93, device="cuda")
    scale = 128 ** -0.5
    o, lse = fa.forward(x.q, x.k, x.v, causal=False, scale=scale)
    exact = oracle.backward(x.q.cpu(), x.k.cpu(), x.v.cpu(), x.do.cpu(), scale, False)
    for _ in range(2):
        got = _noalloc(x.q, x.k, x.v, o, lse, x.do, 1, 4, 4, 513, 513, 128, False, scale, None)
        for name, g, ex in zip(("dq", "dk", "dv"), got, exact):
            assert rel_l2(g, ex) <= GRAD_TOL, name


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    B, Hq, S, d = 1, 32, 4096, 128
    assert fa.fa_bwd_workspace_bytes(B, Hq, S, d, 0) > _scratch_bytes()
    fake = ctypes.c_void_p(0x7F0000000000)  # rejected before any pointer is used
    status = lib.fa_bwd_noalloc(*([fake] * 9), B, Hq, Hq, S, S, d, 1, 0.1, None, None)
    assert status == 5
    assert b"scratch" in lib.fa_last_error()
