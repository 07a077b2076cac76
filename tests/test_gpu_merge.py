"""fa_merge: attention over disjoint key sets, combined through their LSEs.

Parity against the fp64 oracle's attention over the union of the key sets,
with the forward's tolerances (O max-abs 1e-2, LSE max-abs 1e-3), plus the
conventions for rows that saw no key in a part.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_smem_gb300 as fa
import oracle
from attn_inputs import random_inputs
from gpu_helpers import LSE_TOL, O_TOL, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    yield


def _merge(parts, B, Hq, S, d, packed=False):
    o_parts = torch.stack([o for o, _ in parts]).contiguous()
    lse_parts = torch.stack([l for _, l in parts]).contiguous()
    o = torch.empty_like(parts[0][0])
    lse = torch.empty_like(parts[0][1])
    fa.fa_merge(o_parts, lse_parts, len(parts), B, Hq, S, d, packed, o, lse)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 128), (4, 2, 128), (2, 2, 64)])
def test_key_shards_merge_to_full_attention(hq, hkv, d):
    """Non-causal attention over keys split into three uneven shards."""
    x = random_inputs(B=2, Hq=hq, Hkv=hkv, Sq=700, Sk=1000, d=d, seed=300 + hq + d, device="cuda")
    scale = d ** -0.5
    cuts = [0, 200, 450, 1000]
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        k, v = x.k[:, a:b].contiguous(), x.v[:, a:b].contiguous()
        parts.append(fa.forward(x.q, k, v, causal=False, scale=scale))
    o, lse = _merge(parts, 2, hq, 700, d)
    ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), scale, False)
    assert max_abs(o, ro) <= O_TOL
    assert max_abs(lse, rl) <= LSE_TOL


def test_causal_decomposition():
    """Causal attention, rows [a, S): keys [0, a) all visible (non-causal part)
    merged with keys [a, S) under the causal rule (a causal problem of its own)."""
    S, a, d = 1000, 384, 128
    x = random_inputs(B=1, Hq=4, Hkv=2, Sq=S, Sk=S, d=d, seed=310, device="cuda")
    scale = d ** -0.5
    q2 = x.q[:, a:].contiguous()
    p1 = fa.forward(q2, x.k[:, :a].contiguous(), x.v[:, :a].contiguous(), causal=False, scale=scale)
    p2 = fa.forward(q2, x.k[:, a:].contiguous(), x.v[:, a:].contiguous(), causal=True, scale=scale)
    o, lse = _merge([p1, p2], 1, 4, S - a, d)
    ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), scale, True)
    assert max_abs(o, ro[:, a:]) <= O_TOL
    assert max_abs(lse, rl[:, :, a:]) <= LSE_TOL


def test_parts_without_keys_count_zero():
    """A part whose rows saw no key (O = 0, LSE = +inf) leaves the merge
    unchanged; rows with no key in any part get O = 0, LSE = +inf."""
    d = 128
    x = random_inputs(B=1, Hq=2, Hkv=2, Sq=300, Sk=300, d=d, seed=320, device="cuda")
    full = fa.forward(x.q, x.k, x.v, causal=True, scale=0.1)
    empty = (torch.zeros_like(full[0]), torch.full_like(full[1], math.inf))
    o, lse = _merge([empty, full, empty], 1, 2, 300, d)
    assert torch.equal(lse, full[1])
    assert (o.float() - full[0].float()).abs().max().item() <= 2.0 ** -8 * full[0].float().abs().max().item()
    o, lse = _merge([empty, empty], 1, 2, 300, d)
    assert torch.isinf(lse).all() and (lse > 0).all()
    assert (o == 0).all()


def test_packed_layout_and_equal_parts():
    """Packed layout ([T,H,d], LSE [H,T]): two identical parts merge to the same
    O with LSE + ln 2."""
    d = 128
    x = random_inputs(B=None, Hq=2, Hkv=2, Sq=None, Sk=None, d=d, seed=330,
                      lengths=[5, 130, 300], device="cuda")
    T = x.q.shape[0]
    part = fa.forward(x.q, x.k, x.v, causal=True, scale=0.09, cu_seqlens=x.cu_seqlens)
    o, lse = _merge([part, part], 3, 2, T, d, packed=True)
    assert (lse - (part[1] + math.log(2.0))).abs().max().item() <= 1e-5
    assert (o.float() - part[0].float()).abs().max().item() <= 2.0 ** -8 * part[0].float().abs().max().item()


def test_rejects_bad_arguments():
    x = torch.zeros(4, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_merge(x, x, 0, 1, 1, 1, 128, False, x, x)
    assert e.value.status == 1
    with pytest.raises(fa.FAError) as e:
        fa.fa_merge(x, x, 2, 1, 1, 1, 96, False, x, x)
    assert e.value.status == 2


@pytest.mark.parametrize("d", [192, 256])
def test_six_shards_large_head_dim(d):
    """Six uneven key shards (the merge's four-part group plus a remainder)
    at the head dims of the one-tile forward."""
    x = random_inputs(B=1, Hq=2, Hkv=1, Sq=257, Sk=900, d=d, seed=340 + d, device="cuda")
    scale = d ** -0.5
    cuts = [0, 1, 130, 300, 301, 640, 900]
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        k, v = x.k[:, a:b].contiguous(), x.v[:, a:b].contiguous()
        parts.append(fa.forward(x.q, k, v, causal=False, scale=scale))
    o, lse = _merge(parts, 1, 2, 257, d)
    ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), scale, False)
    assert max_abs(o, ro) <= O_TOL
    assert max_abs(lse, rl) <= LSE_TOL
