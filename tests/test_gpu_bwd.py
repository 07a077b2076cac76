"""Backward parity: dQ, dK, dV from the CUDA path against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_smem_gb300 as fa
import oracle
from attn_inputs import random_inputs
from gpu_helpers import GRAD_TOL, guarded, margins_intact, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    yield
    fa.fa_debug_set("grid", 0)
    fa.fa_debug_set("bwd_poly8", 0)


def _dims(x, cu):
    if cu is None:
        B, Sq, Hq, d = x.q.shape
        return B, Hq, x.k.shape[2], Sq, x.k.shape[1], d
    T, Hq, d = x.q.shape
    return cu.numel() - 1, Hq, x.k.shape[1], T, T, d


def _run(x, causal, scale, cu=None):
    B, Hq, Hkv, Sq, Sk, d = _dims(x, cu)
    o, lse = fa.forward(x.q, x.k, x.v, causal=causal, scale=scale, cu_seqlens=cu)
    nbytes = fa.fa_bwd_workspace_bytes(B, Hq, Sq, d, Sq if cu is not None else 0)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")   # garbage on entry
    bufs = [guarded(t.shape, torch.bfloat16, "cuda") for t in (x.q, x.k, x.v)]
    dq, dk, dv = (b[1] for b in bufs)
    fa.fa_bwd(x.q, x.k, x.v, o, lse, x.do, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale, cu,
              ws, nbytes)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    for b, _ in bufs:
        assert margins_intact(b)
    return dq, dk, dv


def _check(x, causal, scale, cu=None, tol=GRAD_TOL):
    dq, dk, dv = _run(x, causal, scale, cu)
    ref = oracle.backward(x.q.cpu(), x.k.cpu(), x.v.cpu(), x.do.cpu(), scale, causal,
                          cu_seqlens=None if cu is None else cu.cpu())
    errs = {}
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert torch.isfinite(got.float()).all(), name
        errs[name] = rel_l2(got, r)
    assert all(e <= tol for e in errs.values()), errs
    return errs


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 63, 64, 127, 128, 129, 300, 513])
def test_dense_shapes(S, causal):
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=S, Sk=S, d=128, seed=1000 + S, device="cuda")
    _check(x, causal, 128 ** -0.5)


@pytest.mark.parametrize("Sq,Sk", [(100, 300), (300, 100), (64, 640)])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_sq_ne_sk(Sq, Sk, causal):
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=Sq, Sk=Sk, d=128, seed=Sq * 7 + Sk, device="cuda")
    _check(x, causal, 0.09)


@pytest.mark.parametrize("hq,hkv", [(8, 1), (8, 2), (6, 3)])
def test_gqa(hq, hkv):
    x = random_inputs(B=2, Hq=hq, Hkv=hkv, Sq=400, Sk=400, d=128, seed=hq * 31 + hkv, device="cuda")
    _check(x, True, 128 ** -0.5)


@pytest.mark.parametrize("lengths", [[1, 127, 128, 129, 300], [700], [5, 0, 600, 1], [64] * 6])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen(lengths, causal):
    x = random_inputs(B=None, Hq=4, Hkv=2, Sq=None, Sk=None, d=128, seed=sum(lengths) + 2,
                      lengths=lengths, device="cuda")
    _check(x, causal, 128 ** -0.5, cu=x.cu_seqlens)


def test_gqa_matches_repeated_kv():
    """dK/dV of a KV head equal the sum over its query heads of the MHA gradients."""
    x = random_inputs(B=1, Hq=4, Hkv=1, Sq=384, Sk=384, d=128, seed=77, device="cuda")
    dq, dk, dv = _run(x, True, 0.1)
    xr = type(x)(x.q, x.k.repeat_interleave(4, dim=2).contiguous(),
                 x.v.repeat_interleave(4, dim=2).contiguous(), x.do, None, None, None)
    dq2, dk2, dv2 = _run(xr, True, 0.1)
    assert (dq.float() - dq2.float()).abs().max().item() <= 1e-2 * dq2.float().abs().max().item()
    for a, b in ((dk, dk2), (dv, dv2)):
        s = b.float().sum(dim=2, keepdim=True)
        assert (a.float() - s).abs().max().item() <= 2e-2 * s.abs().max().item()


def test_schedule_permutation():
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=700, Sk=700, d=128, seed=78, device="cuda")
    a = _run(x, True, 0.1)
    fa.fa_debug_set("grid", 5)
    b = _run(x, True, 0.1)
    fa.fa_debug_set("grid", 0)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])     # dK, dV: no atomics
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("poly8", [2, 4])
def test_poly_exp_split(poly8):
    fa.fa_debug_set("bwd_poly8", poly8)
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=500, Sk=500, d=128, seed=79, device="cuda")
    _check(x, True, 128 ** -0.5)
    fa.fa_debug_set("bwd_poly8", 0)


def test_head_dim_64_backward_is_reported_unsupported():
    x = random_inputs(B=1, Hq=2, Hkv=2, Sq=128, Sk=128, d=64, seed=80, device="cuda")
    with pytest.raises(fa.FAError) as e:
        _run(x, False, 0.125)
    assert e.value.status == 2
