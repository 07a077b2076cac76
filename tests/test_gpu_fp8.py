"""FP8 (e4m3) path: quantization and forward against the oracle.

* fa_quantize_fp8: codes and scales bit-exact against the oracle's quantizer
  (both sides take every decision in float32: amax, amax / 448, 1 / scale,
  x * (1 / scale), round to nearest even with saturation).
* fa_fwd_fp8 against exact fp64 attention over the dequantized inputs:
  - LSE max-abs <= 1e-3: the scores are exact sums of code products
    accumulated in fp32, as in the bf16 forward;
  - O rel-L2 <= 5e-2 (per head): the kernel rounds each softmax weight to
    e4m3 (3 mantissa bits, relative rounding error <= 2^-4, so an RMS of at
    most 2^-4 / sqrt(3) = 3.6% per weight). The output is a weighted sum of
    V rows, so independent relative errors in the weights give an output
    error whose RMS is at most that of the weights, 3.6% of the RMS output;
    5e-2 leaves headroom for bf16 output rounding. A structural error (a
    wrong block scale, a dropped key block, a transposed operand) is off by
    tens of percent or more;
  - O element by element (so that one badly wrong row cannot hide under the
    per-head norm): a weight in e4m3's normal range is off by at most 2^-4 of
    itself; the kernel stores 2^7 times the weight, so one below the normal
    range is off by at most half the smallest subnormal step, 2^-10, i.e.
    2^-17 of the row's largest weight; the row sum is taken over the unrounded
    weights. Hence
        |O - O*|_ic <= (2^-4 + 2^-8) sum_j P_ij |V_jc|
                       + 2^-17 max_j P_ij sum_{j visible} |V_jc| + ulp_bf16 / 2,
    with P the exact softmax weights; 2^-8 covers the fp32 accumulation of
    the scores and of P V. Both sums come from the oracle (attention over |V|,
    and with Q = 0 the mean of the visible |V| rows), max_j P_ij from its row
    maxima, exp(m_i - LSE_i);
  - Q = 0 makes every weight exactly 1 (2^7 in the kernel, exact in e4m3), so
    O is the plain mean of the visible V rows: checked to 4e-3 max-abs (bf16
    output rounding).
"""
import numpy as np
import pytest
import torch

import exact_attention_smem_gb300 as fa
from oracle import fp8_e4m3 as f8
from attn_inputs import random_inputs
from gpu_helpers import LSE_TOL, max_abs

pytestmark = pytest.mark.gpu

O_REL_L2_FP8 = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _dev():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    yield
    assert fa.fa_get_device_error(clear=True) == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [1, 127, 300])
def test_quantize_rows_bit_exact(S, d):
    g = torch.Generator().manual_seed(10 + S + d)
    x = (torch.randn(2, S, 3, d, generator=g) * torch.rand(1, S, 3, 1, generator=g) * 4)
    x = x.to(torch.bfloat16)
    if S > 128:
        x[1, 128:256, 2] = 0                          # an all-zero block
    codes, scales = fa.quantize_fp8(x.cuda(), 0)
    torch.cuda.synchronize()
    rc, rs = f8.quantize_row_blocks(x.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [1, 37, 300, 1000])
def test_quantize_v_bit_exact(S, d):
    g = torch.Generator().manual_seed(20 + S + d)
    x = (torch.randn(2, S, 3, d, generator=g) * 3).to(torch.bfloat16)
    codes, scales = fa.quantize_fp8(x.cuda(), 1)
    torch.cuda.synchronize()
    rc, rs = f8.quantize_v_transposed(x.float().numpy())
    assert codes.shape == rc.shape
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


def _bf16_half_ulp(x):
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8)


def _check_elementwise(o, codes, scale, causal, heads=None, seqs=None):
    """Element-wise bound on the FP8 forward's O (module docstring); o is the
    kernel's O as float [B, Sq, Hq, d], codes = (q8, qs, k8, ks, v8, vs) as
    numpy arrays. Returns the largest error / bound ratio (must be <= 1)."""
    q8, qs, k8, ks, v8, vs = codes
    ro, rl, rm = f8.forward_fp8(q8, qs, k8, ks, v8, vs, scale, causal, heads=heads, seqs=seqs,
                                return_max=True)
    v_abs = v8 & np.uint8(0x7F)                       # e4m3 sign bit cleared: |V|
    a, _ = f8.forward_fp8(q8, qs, k8, ks, v_abs, vs, scale, causal, heads=heads, seqs=seqs)
    mean_abs, _ = f8.forward_fp8(np.zeros_like(q8), qs, k8, ks, v_abs, vs, scale, causal,
                                 heads=heads, seqs=seqs)
    B, Sq, Hq, d = ro.shape
    Sk = k8.shape[1]
    i = np.arange(Sq)
    n_vis = np.clip(i + 1 + Sk - Sq, 0, Sk) if causal else np.full(Sq, Sk)
    sum_abs = mean_abs * n_vis[None, :, None, None]
    with np.errstate(invalid="ignore"):
        p_max = np.where(np.isfinite(rl), np.exp(rm - rl), 0.0)       # [B, Hq, Sq]
    p_max = p_max.transpose(0, 2, 1)[..., None]
    bound = ((2.0 ** -4 + 2.0 ** -8) * a + 2.0 ** -17 * p_max * sum_abs +
             _bf16_half_ulp(np.maximum(np.abs(o), np.abs(ro))) + 1e-6)
    sel = ~np.isnan(ro)
    ratio = np.abs(o - ro)[sel] / bound[sel]
    assert np.all(np.isfinite(o[sel]))
    return float(ratio.max()) if ratio.size else 0.0


def _fp8_case(B, Hq, Hkv, Sq, Sk, causal, seed, zero_q=False):
    x = random_inputs(B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, d=128, seed=seed, device="cuda")
    q = torch.zeros_like(x.q) if zero_q else x.q
    q8, qs = fa.quantize_fp8(q, 0)
    k8, ks = fa.quantize_fp8(x.k, 0)
    v8, vs = fa.quantize_fp8(x.v, 1)
    scale = 128 ** -0.5
    o, lse = fa.forward_fp8(q8, qs, k8, ks, v8, vs, causal=causal, scale=scale)
    torch.cuda.synchronize()
    codes = tuple(t.cpu().numpy() for t in (q8, qs, k8, ks, v8, vs))
    ro, rl = f8.forward_fp8(*codes, scale, causal)
    o = o.float().cpu().numpy()
    assert _check_elementwise(o, codes, scale, causal) <= 1.0
    return o, lse.cpu(), ro, rl


def _rel_l2_per_head(o, ro):
    worst = 0.0
    for h in range(o.shape[2]):
        a, b = o[:, :, h], ro[:, :, h]
        fin = np.isfinite(b)
        num = np.linalg.norm((a - b)[fin])
        den = np.linalg.norm(b[fin])
        if den > 0:
            worst = max(worst, num / den)
    return worst


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk", [(2, 4, 2, 300, 300), (1, 2, 2, 200, 700),
                                            (1, 2, 1, 700, 200), (1, 2, 2, 1024, 1024)])
def test_fp8_forward_parity(B, Hq, Hkv, Sq, Sk, causal):
    o, lse, ro, rl = _fp8_case(B, Hq, Hkv, Sq, Sk, causal, seed=40 + Sq + Sk + causal)
    assert max_abs(lse, rl) <= LSE_TOL
    assert _rel_l2_per_head(o, ro) <= O_REL_L2_FP8
    # rows with no visible key: O = 0, LSE = +inf
    empty = ~np.isfinite(rl)
    if empty.any():
        ln = lse.numpy()
        assert np.all(np.isinf(ln[empty])) and np.all(ln[empty] > 0)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_uniform_weights_exact(causal):
    o, lse, ro, rl = _fp8_case(1, 2, 2, 384, 500, causal, seed=77, zero_q=True)
    assert max_abs(lse, rl) <= LSE_TOL
    fin = np.isfinite(ro)
    assert np.abs(o[fin] - ro[fin]).max() <= 4e-3


def test_fp8_rejects_bad_arguments():
    x = torch.zeros(16, device="cuda", dtype=torch.uint8)
    f = torch.zeros(4, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_fp8(x, x, x, f, f, f, x, f, 1, 2, 2, 16, 16, 64, 0, 0.1)
    assert e.value.status == 2
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_fp8(x, x, x, f, f, f, x, f, 1, 3, 2, 16, 16, 128, 0, 0.1)
    assert e.value.status == 1
    with pytest.raises(fa.FAError) as e:
        fa.fa_quantize_fp8(x, 1, 16, 1, 128, 2, x, f)
    assert e.value.status == 1


@pytest.mark.parametrize("poly8", [2, 4])
def test_fp8_forward_polynomial_exp2(poly8):
    """Some exponentials from the FMA-pipe polynomial (relative error ~1e-7,
    far below the e4m3 rounding of the weights): same bounds."""
    fa.fa_debug_set("fp8_poly8", poly8)
    try:
        o, lse, ro, rl = _fp8_case(2, 4, 2, 300, 700, True, seed=90 + poly8)
    finally:
        fa.fa_debug_set("fp8_poly8", 0)
    assert max_abs(lse, rl) <= LSE_TOL
    assert _rel_l2_per_head(o, ro) <= O_REL_L2_FP8


@pytest.mark.parametrize("name", ["long_s32768_causal", "gqa_s8192_causal"])
def test_fp8_full_size_parity(name):
    """The workloads `bench.py --fp8` times, at full size in its launch
    configuration; the oracle checks query heads {0, last} (long) or KV group 0
    of the first and last batch entries (GQA)."""
    from attn_inputs import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    x = make_inputs(w, "cuda")
    q8, qs = fa.quantize_fp8(x.q, 0)
    k8, ks = fa.quantize_fp8(x.k, 0)
    v8, vs = fa.quantize_fp8(x.v, 1)
    del x
    o, lse = fa.forward_fp8(q8, qs, k8, ks, v8, vs, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    if name == "gqa_s8192_causal":
        heads, seqs = list(range(w.Hq // w.Hkv)), [0, w.B - 1]
    else:
        heads, seqs = [0, w.Hq - 1], None
    codes = tuple(t.cpu().numpy() for t in (q8, qs, k8, ks, v8, vs))
    ro, rl = f8.forward_fp8(*codes, w.scale, True, heads=heads, seqs=seqs)
    bsel = list(range(w.B)) if seqs is None else seqs
    lse_c = lse.cpu()
    e_lse = max_abs(lse_c[bsel][:, heads], rl[bsel][:, heads])
    o_all = o.float().cpu().numpy()
    o_c = o_all[bsel][:, :, heads]
    e_o = _rel_l2_per_head(o_c, ro[bsel][:, :, heads])
    ratio = _check_elementwise(o_all, codes, w.scale, True, heads=heads, seqs=seqs)
    print(f"\nfp8 {name}: LSE max-abs {e_lse:.2e}, O rel-L2 (worst head) {e_o:.2e}, "
          f"element-wise error / bound {ratio:.3f}")
    assert e_lse <= LSE_TOL
    assert e_o <= O_REL_L2_FP8
    assert ratio <= 1.0


@pytest.mark.parametrize("tau", [0.0, 1.0])
def test_fp8_forward_rescale_threshold(tau):
    """Thresholds other than the default 1.5 (the largest weight the kernel
    stores, 2^(7 + tau), stays below e4m3's 448 for any tau <= 1.5): same
    bounds."""
    fa.fa_debug_set("fp8_tau", tau)
    try:
        o, lse, ro, rl = _fp8_case(2, 4, 2, 300, 1000, True, seed=120 + int(tau))
    finally:
        fa.fa_debug_set("fp8_tau", 1.5)
    assert max_abs(lse, rl) <= LSE_TOL
    assert _rel_l2_per_head(o, ro) <= O_REL_L2_FP8
    with pytest.raises(fa.FAError):
        fa.fa_debug_set("fp8_tau", 2.0)


def test_fp8_output_16_byte_aligned_only():
    """O at an address that is 16- but not 32-byte aligned: the same values,
    bit for bit, as into an aligned buffer (whole tiles leave through TMA
    stores, the rest per thread)."""
    x = random_inputs(B=2, Hq=2, Hkv=2, Sq=300, Sk=300, d=128, seed=5, device="cuda")
    q8, qs = fa.quantize_fp8(x.q, 0)
    k8, ks = fa.quantize_fp8(x.k, 0)
    v8, vs = fa.quantize_fp8(x.v, 1)
    ref, ref_lse = fa.forward_fp8(q8, qs, k8, ks, v8, vs, causal=True, scale=128 ** -0.5)
    raw = torch.full((x.q.numel() + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = raw[8:].view(x.q.shape)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty_like(ref_lse)
    fa.forward_fp8(q8, qs, k8, ks, v8, vs, causal=True, scale=128 ** -0.5, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error(clear=True) == 0
    assert torch.isnan(raw[:8].float()).all()
    assert torch.equal(o, ref) and torch.equal(lse, ref_lse)
