"""Packed sequences with separate query and key boundaries (fa_fwd_varlen,
fa_bwd_varlen): prefill over cached keys (more keys than queries), fewer keys
than queries (bottom-right causal leaves early rows without keys), equal
counts, and sequences with no keys, at head dims 64, 128, 192 and 256; and
300 packed sequences, more boundaries than the kernels keep in shared memory.
Parity against the fp64 oracle with the tolerances of the other tests."""
import pytest
import torch

import exact_attention_smem_gb300 as fa
import oracle
from attn_inputs import random_inputs
from gpu_helpers import GRAD_TOL, LSE_TOL, O_TOL, max_abs, rel_l2

pytestmark = pytest.mark.gpu

CASES = [
    ([5, 130, 300, 64, 1], [5, 400, 300, 1000, 0]),
    ([257, 3, 128], [129, 700, 128]),
    ([1], [2000]),
]


@pytest.fixture(scope="module", autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    yield
    fa.fa_debug_set("bwd_mode", 1)


@pytest.mark.parametrize("bwd_mode", [1, 0])
@pytest.mark.parametrize("d,hq,hkv", [(128, 4, 2), (64, 2, 2), (192, 4, 2), (256, 2, 1)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_separate_boundaries(case, causal, d, hq, hkv, bwd_mode):
    if bwd_mode == 0 and d != 128:
        pytest.skip("the one-pass form supports d=128 only")
    lq, lk = CASES[case]
    fa.fa_debug_set("bwd_mode", bwd_mode)
    x = random_inputs(B=None, Hq=hq, Hkv=hkv, Sq=None, Sk=None, d=d, seed=400 + case * 7 + d,
                      lengths=lq, lengths_k=lk, device="cuda")
    scale = d ** -0.5
    cu, cuk = x.cu_seqlens, x.cu_seqlens_k
    o, lse = fa.forward(x.q, x.k, x.v, causal=causal, scale=scale, cu_seqlens=cu, cu_seqlens_k=cuk)
    grads = fa.backward(x.q, x.k, x.v, o, lse, x.do, causal=causal, scale=scale, cu_seqlens=cu,
                        cu_seqlens_k=cuk)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    qc, kc, vc, doc = (t.cpu() for t in (x.q, x.k, x.v, x.do))
    ro, rl = oracle.forward(qc, kc, vc, scale, causal, cu_seqlens=cu.cpu(), cu_seqlens_k=cuk.cpu())
    assert max_abs(o, ro) <= O_TOL
    assert max_abs(lse, rl) <= LSE_TOL
    ref = oracle.backward(qc, kc, vc, doc, scale, causal, cu_seqlens=cu.cpu(),
                          cu_seqlens_k=cuk.cpu())
    errs = {n: rel_l2(g, r) for n, g, r in zip(("dq", "dk", "dv"), grads, ref)}
    assert all(e <= GRAD_TOL for e in errs.values()), errs


def test_rejects_missing_key_list():
    x = random_inputs(B=None, Hq=2, Hkv=2, Sq=None, Sk=None, d=128, seed=450, lengths=[10],
                      lengths_k=[20], device="cuda")
    o = torch.empty_like(x.q)
    lse = torch.empty(2, 10, dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_varlen(x.q, x.k, x.v, o, lse, 1, 2, 2, 10, 20, 128, True, 0.1, x.cu_seqlens, None)
    assert e.value.status == 1


@pytest.mark.parametrize("separate_keys", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_many_sequences_read_boundaries_from_global_memory(causal, separate_keys):
    """300 packed sequences: more boundaries than the kernels keep in shared
    memory (forward 256 entries, backward 200; separate key lists take two
    entries per sequence), so every role reads them from global memory."""
    g = torch.Generator().manual_seed(7)
    lq = [int(x) for x in torch.randint(0, 40, (300,), generator=g)]
    lk = [int(x) for x in torch.randint(0, 60, (300,), generator=g)] if separate_keys else None
    d, hq, hkv = 128, 2, 1
    x = random_inputs(B=None, Hq=hq, Hkv=hkv, Sq=None, Sk=None, d=d, seed=77, lengths=lq,
                      lengths_k=lk, device="cuda")
    scale = d ** -0.5
    cu, cuk = x.cu_seqlens, x.cu_seqlens_k
    o, lse = fa.forward(x.q, x.k, x.v, causal=causal, scale=scale, cu_seqlens=cu, cu_seqlens_k=cuk)
    grads = fa.backward(x.q, x.k, x.v, o, lse, x.do, causal=causal, scale=scale, cu_seqlens=cu,
                        cu_seqlens_k=cuk)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    qc, kc, vc, doc = (t.cpu() for t in (x.q, x.k, x.v, x.do))
    cuk_c = None if cuk is None else cuk.cpu()
    ro, rl = oracle.forward(qc, kc, vc, scale, causal, cu_seqlens=cu.cpu(), cu_seqlens_k=cuk_c)
    assert max_abs(o, ro) <= O_TOL
    assert max_abs(lse, rl) <= LSE_TOL
    ref = oracle.backward(qc, kc, vc, doc, scale, causal, cu_seqlens=cu.cpu(), cu_seqlens_k=cuk_c)
    errs = {n: rel_l2(g_, r) for n, g_, r in zip(("dq", "dk", "dv"), grads, ref)}
    assert all(e <= GRAD_TOL for e in errs.values()), errs
