"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import exact_attention_smem_gb300 as fa
import oracle
from attn_inputs import WORKLOADS, make_inputs, random_inputs
from gpu_helpers import LSE_TOL, O_TOL, guarded, margins_intact, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    yield
    fa.fa_debug_set("grid", 0)
    fa.fa_debug_set("tau", 0)
    fa.fa_debug_set("poly8", 0)
    fa.fa_debug_set("fwd_split_q", -1)


def _run(x, causal, scale, cu=None):
    """Forward into sentinel-guarded outputs; returns (o, lse) and checks the guards."""
    q = x.q
    if cu is None:
        B, Sq, Hq, d = q.shape
        lse_shape = (B, Hq, Sq)
    else:
        T, Hq, d = q.shape
        B, Sq = cu.numel() - 1, T
        lse_shape = (Hq, T)
    Sk = x.k.shape[1] if cu is None else x.k.shape[0]
    obuf, o = guarded(q.shape, torch.bfloat16, q.device)
    lbuf, lse = guarded(lse_shape, torch.float32, q.device)
    fa.fa_fwd(q, x.k, x.v, o, lse, B, Hq, x.k.shape[-2], Sq, Sk, d, causal, scale, cu)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    assert margins_intact(obuf) and margins_intact(lbuf)
    return o, lse


def _check(x, causal, scale, cu=None, o_tol=O_TOL):
    o, lse = _run(x, causal, scale, cu)
    ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), scale, causal,
                            cu_seqlens=None if cu is None else cu.cpu())
    eo, el = max_abs(o, ro), max_abs(lse, rl)
    assert np.isfinite(o.float().cpu().numpy()).all()
    assert eo <= o_tol, f"O max-abs {eo}"
    assert el <= LSE_TOL, f"LSE max-abs {el}"
    return o, lse, eo, el


def test_workload_fwd_small_d64():
    w = WORKLOADS["fwd_small_d64"]
    x = make_inputs(w, "cuda")
    _check(x, w.causal, w.scale)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 17, 128, 129, 255, 256, 257, 700])
def test_dense_shapes(S, causal, d):
    x = random_inputs(B=2, Hq=3, Hkv=3, Sq=S, Sk=S, d=d, seed=S * 3 + d, device="cuda")
    _check(x, causal, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("Sq,Sk", [(100, 300), (300, 100), (256, 513), (1, 700)])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_sq_ne_sk(Sq, Sk, causal):
    x = random_inputs(B=2, Hq=2, Hkv=1, Sq=Sq, Sk=Sk, d=128, seed=Sq + Sk, device="cuda")
    o, lse, _, _ = _check(x, causal, 0.09)
    if causal and Sq > Sk:
        # rows that see no key: O = 0, LSE = +inf
        n_empty = Sq - Sk
        assert torch.all(o[:, :n_empty] == 0)
        assert torch.all(torch.isinf(lse[:, :, :n_empty]))


@pytest.mark.parametrize("hq,hkv", [(8, 1), (8, 2), (6, 3)])
def test_gqa(hq, hkv):
    x = random_inputs(B=2, Hq=hq, Hkv=hkv, Sq=400, Sk=400, d=128, seed=hq * 10 + hkv, device="cuda")
    _check(x, True, 128 ** -0.5)


@pytest.mark.parametrize("lengths", [[1, 127, 128, 129, 300], [700], [5, 0, 600, 1], [256] * 5])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen(lengths, causal):
    x = random_inputs(B=None, Hq=4, Hkv=2, Sq=None, Sk=None, d=128, seed=sum(lengths) + 1,
                      lengths=lengths, device="cuda")
    _check(x, causal, 128 ** -0.5, cu=x.cu_seqlens)


def test_varlen_equals_per_sequence_dense_bitwise():
    lengths = [300, 129, 1000]
    x = random_inputs(B=None, Hq=2, Hkv=2, Sq=None, Sk=None, d=128, seed=5, lengths=lengths,
                      device="cuda")
    o, lse = _run(x, True, 0.1, x.cu_seqlens)
    start = 0
    for L in lengths:
        sl = slice(start, start + L)
        xs = type(x)(x.q[None, sl], x.k[None, sl], x.v[None, sl], x.do[None, sl], None, None, None)
        od, ld = _run(xs, True, 0.1)
        assert torch.equal(o[sl], od[0])
        assert torch.equal(lse[:, sl], ld[0])
        start += L


def test_v_all_ones_gives_ones():
    x = random_inputs(B=1, Hq=2, Hkv=2, Sq=600, Sk=600, d=128, seed=9, device="cuda", std=2.0)
    x.v.fill_(1.0)
    o, _ = _run(x, True, 0.2)
    assert (o.float() - 1).abs().max().item() <= 2 ** -8


def test_causal_row0_is_v0_exactly():
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=300, Sk=300, d=128, seed=10, device="cuda")
    o, lse = _run(x, True, 0.1)
    assert torch.equal(o[:, 0], x.v[:, 0])


def test_schedule_permutation_is_bitwise_invisible():
    x = random_inputs(B=3, Hq=4, Hkv=4, Sq=900, Sk=900, d=128, seed=11, device="cuda")
    o1, l1 = _run(x, True, 0.1)
    for g in (1, 7, 64):
        fa.fa_debug_set("grid", g)
        o2, l2 = _run(x, True, 0.1)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    fa.fa_debug_set("grid", 0)


@pytest.mark.parametrize("tau", [0.0, 1.0, 3.0, 8.0])
def test_rescale_threshold_keeps_parity(tau):
    fa.fa_debug_set("tau", tau)
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=1024, Sk=1024, d=128, seed=12, device="cuda", std=1.5)
    _check(x, True, 128 ** -0.5)
    fa.fa_debug_set("tau", 0)


@pytest.mark.parametrize("poly8", [2, 4])
def test_poly_exp_split_keeps_parity(poly8):
    fa.fa_debug_set("poly8", poly8)
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=700, Sk=700, d=128, seed=13, device="cuda")
    _check(x, True, 128 ** -0.5)
    fa.fa_debug_set("poly8", 0)


@pytest.mark.parametrize("d", [64, 128])
def test_output_16_byte_aligned_only(d):
    """O at an address that is 16- but not 32-byte aligned (the C ABI asks for
    16): whole tiles still leave through TMA stores, the rest per thread."""
    x = random_inputs(B=2, Hq=3, Hkv=3, Sq=300, Sk=300, d=d, seed=17 + d, device="cuda")
    B, Sq, Hq, _ = x.q.shape
    raw = torch.full((x.q.numel() + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = raw[8:].view(x.q.shape)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    fa.fa_fwd(x.q, x.k, x.v, o, lse, B, Hq, Hq, Sq, Sq, d, True, d ** -0.5, None)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    assert torch.isnan(raw[:8].float()).all()                # nothing written before O
    ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), d ** -0.5, True)
    assert max_abs(o, ro) <= O_TOL
    assert max_abs(lse, rl) <= LSE_TOL


@pytest.mark.parametrize("case", ["causal", "noncausal_d64", "sq_ne_sk", "gqa", "packed",
                                  "long_units"])
def test_split_q_barriers_bitwise_invisible(case):
    """The two ways of loading a unit's two Q tiles (one barrier pair for both,
    or one pair per tile so that tile 0's next Q loads early) give the same
    bits, on dense, GQA and packed layouts (the automatic choice uses the
    per-tile form only for dense layouts with at most 4096 keys), and the
    per-tile form matches the oracle."""
    cu = None
    if case == "causal":
        x, causal = random_inputs(B=2, Hq=4, Hkv=4, Sq=700, Sk=700, d=128, seed=95,
                                  device="cuda"), True
    elif case == "noncausal_d64":
        x, causal = random_inputs(B=2, Hq=4, Hkv=4, Sq=300, Sk=300, d=64, seed=96,
                                  device="cuda"), False
    elif case == "sq_ne_sk":
        x, causal = random_inputs(B=2, Hq=2, Hkv=2, Sq=300, Sk=900, d=128, seed=97,
                                  device="cuda"), True
    elif case == "gqa":
        x, causal = random_inputs(B=1, Hq=8, Hkv=2, Sq=513, Sk=513, d=128, seed=98,
                                  device="cuda"), True
    elif case == "packed":
        x = random_inputs(B=None, Hq=4, Hkv=4, Sq=None, Sk=None, d=128, seed=99,
                          lengths=[1, 127, 128, 129, 300, 700, 256], device="cuda")
        causal, cu = True, x.cu_seqlens
    else:   # a few units of many blocks each (S = 4096: the largest automatic case)
        x, causal = random_inputs(B=1, Hq=2, Hkv=2, Sq=4096, Sk=4096, d=128, seed=100,
                                  device="cuda"), True
    scale = 1.0 / math.sqrt(x.q.shape[-1])
    outs = []
    try:
        for mode in (0, 1):
            fa.fa_debug_set("fwd_split_q", mode)
            outs.append(_run(x, causal, scale, cu))
    finally:
        fa.fa_debug_set("fwd_split_q", -1)
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    if case != "long_units":
        ro, rl = oracle.forward(x.q.cpu(), x.k.cpu(), x.v.cpu(), scale, causal,
                                cu_seqlens=None if cu is None else cu.cpu())
        assert max_abs(outs[1][0], ro) <= O_TOL and max_abs(outs[1][1], rl) <= LSE_TOL
