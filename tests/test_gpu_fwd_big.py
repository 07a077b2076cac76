"""Forward parity for head dims 192 and 256 (one query tile per CTA, 64-key
blocks, S two blocks ahead): the fp64 oracle with the forward's tolerances
(O max-abs 1e-2, LSE max-abs 1e-3)."""
import pytest
import torch

import exact_attention_smem_gb300 as fa
import oracle
from attn_inputs import random_inputs
from gpu_helpers import LSE_TOL, O_TOL, guarded, margins_intact, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    yield
    fa.fa_debug_set("tau", 0)


def _check(x, causal, scale, cu=None, cuk=None):
    if cu is None:
        B, Sq, Hq, d = x.q.shape
        shape_lse = (B, Hq, Sq)
    else:
        Sq, Hq, d = x.q.shape
        shape_lse = (Hq, Sq)
    bo, o = guarded(x.q.shape, torch.bfloat16, "cuda")
    lse = torch.empty(shape_lse, dtype=torch.float32, device="cuda")
    fa.forward(x.q, x.k, x.v, causal=causal, scale=scale, cu_seqlens=cu, cu_seqlens_k=cuk,
               out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    assert margins_intact(bo)
    ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), scale, causal,
                            cu_seqlens=None if cu is None else cu.cpu(),
                            cu_seqlens_k=None if cuk is None else cuk.cpu())
    assert max_abs(o, ro) <= O_TOL
    assert max_abs(lse, rl) <= LSE_TOL
    return o, lse


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 63, 64, 65, 127, 129, 300, 700])
def test_dense_shapes(S, causal, d):
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=S, Sk=S, d=d, seed=500 + S + d, device="cuda")
    _check(x, causal, d ** -0.5)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("Sq,Sk", [(100, 300), (300, 100), (64, 640)])
def test_sq_ne_sk(Sq, Sk, d):
    x = random_inputs(B=2, Hq=4, Hkv=2, Sq=Sq, Sk=Sk, d=d, seed=Sq * 3 + Sk + d, device="cuda")
    _check(x, True, 0.07)


@pytest.mark.parametrize("d", [192, 256])
def test_packed_and_separate_key_boundaries(d):
    x = random_inputs(B=None, Hq=4, Hkv=1, Sq=None, Sk=None, d=d, seed=520 + d,
                      lengths=[1, 64, 129, 300], device="cuda")
    _check(x, True, d ** -0.5, cu=x.cu_seqlens)
    y = random_inputs(B=None, Hq=2, Hkv=2, Sq=None, Sk=None, d=d, seed=530 + d,
                      lengths=[5, 130, 64], lengths_k=[300, 0, 64], device="cuda")
    _check(y, True, d ** -0.5, cu=y.cu_seqlens, cuk=y.cu_seqlens_k)


@pytest.mark.parametrize("tau", [0.0, 3.0])
def test_rescale_under_growing_scores(tau):
    """Keys scaled up along the sequence make the running row max grow block
    after block, so O is rescaled while S runs ahead of the PV accumulation."""
    fa.fa_debug_set("tau", tau)
    d, S = 256, 640
    x = random_inputs(B=1, Hq=2, Hkv=2, Sq=S, Sk=S, d=d, seed=540, device="cuda")
    ramp = torch.linspace(0.2, 3.0, S, device="cuda").view(1, S, 1, 1)
    k = (x.k.float() * ramp).to(torch.bfloat16).contiguous()
    y = type(x)(x.q, k, x.v, x.do, None, None, None)
    for causal in (False, True):
        _check(y, causal, d ** -0.5)
    fa.fa_debug_set("tau", 0)


def test_merge_at_head_dim_256():
    d = 256
    x = random_inputs(B=1, Hq=2, Hkv=2, Sq=300, Sk=700, d=d, seed=550, device="cuda")
    parts = [fa.forward(x.q, x.k[:, a:b].contiguous(), x.v[:, a:b].contiguous(), causal=False,
                        scale=0.06) for a, b in ((0, 250), (250, 700))]
    o_parts = torch.stack([o for o, _ in parts]).contiguous()
    l_parts = torch.stack([l for _, l in parts]).contiguous()
    o, lse = torch.empty_like(parts[0][0]), torch.empty_like(parts[0][1])
    fa.fa_merge(o_parts, l_parts, 2, 1, 2, 300, d, False, o, lse)
    torch.cuda.synchronize()
    ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), 0.06, False)
    assert max_abs(o, ro) <= O_TOL and max_abs(lse, rl) <= LSE_TOL
