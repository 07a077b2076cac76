"""FP8 (e4m3) quantization and the FP8 attention forward's definition.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``): only
``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import it; the CUDA path never does.

The FlashAttention-4 pages name the low-precision lineage only by the title of
FlashAttention-3 ("Fast and Accurate Attention with Asynchrony and Low
Precision", reference lists of the pages); they give no FP8 algorithm. So every
choice below is a stated reading, the plainest one the rest supports:

* e4m3 is the 8-bit format with 1 sign bit, 4 exponent bits (bias 7) and 3
  mantissa bits: normal values (1 + m/8) * 2^(e-7) for e in 1..15 (except
  e = 15, m = 7, the NaN code), subnormals (m/8) * 2^-6 for e = 0. No
  infinities; the largest finite value is 448. Encoding rounds to the nearest
  representable value, ties to the even code, and saturates to +-448.
* Q and K are quantized per (sequence, head, block of 128 rows): scale =
  amax / 448 over the block's rows and all d columns (1 when amax = 0), code =
  e4m3(x * r) with r = 1 / scale rounded to float32 once per block. V is
  quantized per (sequence, head) over all its rows, and stored transposed
  ([B, H, d, S_pad], keys contiguous, S_pad = S rounded up to 16, the pad
  written as zero codes). scale, r and x * r are each rounded to float32
  (IEEE division and multiply), so the GPU makes the same decisions.
* The FP8 forward is exact attention over the dequantized inputs
  q_hat = decode(code) * scale (and likewise k_hat, v_hat). The kernel rounds
  the softmax weights to e4m3 before its P V product; that rounding is the one
  approximation beyond the definition, and the parity tests bound it.

Parity pins (tests/test_oracle_fp8.py): the format's fixed points (448, the
smallest normal and subnormal, one, zero), ties to even, saturation, a
round trip over every finite code, monotonicity, and brute force nearest-value
search on random inputs.
"""
from __future__ import annotations

import numpy as np

from .attention_fp64 import attend_head as _attend_head

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


# the 127 non-negative finite values, increasing with the code (0x00 .. 0x7E)
_POS = e4m3_decode(np.arange(127, dtype=np.uint8))


def e4m3_encode(x) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to the even code), saturating at
    +-448; NaN -> 0x7F. Works on float32 or float64 input, elementwise."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    a_sat = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_POS, a_sat, side="left")       # first value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a_sat - _POS[lo]
    d_hi = _POS[hi] - a_sat
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(_POS[hi] == a_sat, hi, np.where(take_hi, hi, lo)).astype(np.int64)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def _f32(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float32)


def quantize_row_blocks(x, block: int = BLOCK):
    """Q or K [B, S, H, d] -> (codes uint8 [B, S, H, d], scales float32 [B, H, nblk])."""
    x = _f32(x)
    B, S, H, d = x.shape
    nblk = (S + block - 1) // block
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.ones((B, H, nblk), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            for i in range(nblk):
                blk = x[b, i * block:(i + 1) * block, h, :]
                amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
                s = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
                scales[b, h, i] = s
                codes[b, i * block:(i + 1) * block, h, :] = e4m3_encode(blk * (np.float32(1) / s))
    return codes, scales


def v_pad(S: int) -> int:
    return (S + 15) // 16 * 16


def quantize_v_transposed(v):
    """V [B, S, H, d] -> (codes uint8 [B, H, d, S_pad] (keys contiguous, pad = 0),
    scales float32 [B, H])."""
    v = _f32(v)
    B, S, H, d = v.shape
    codes = np.zeros((B, H, d, v_pad(S)), dtype=np.uint8)
    scales = np.ones((B, H), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            blk = v[b, :, h, :]
            amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
            s = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
            scales[b, h] = s
            codes[b, h, :, :S] = e4m3_encode(blk * (np.float32(1) / s)).T
    return codes, scales


def dequantize_row_blocks(codes, scales, block: int = BLOCK):
    """Inverse view of quantize_row_blocks: float64 [B, S, H, d]."""
    vals = e4m3_decode(codes)
    S = vals.shape[1]
    rep = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=2)[:, :, :S]  # [B, H, S]
    return vals * rep.transpose(0, 2, 1)[..., None]


def dequantize_v_transposed(codes, scales, S: int):
    """Inverse view of quantize_v_transposed: float64 [B, S, H, d]."""
    vals = e4m3_decode(np.asarray(codes)[..., :S])           # [B, H, d, S]
    vals = vals * np.asarray(scales, dtype=np.float64)[:, :, None, None]
    return vals.transpose(0, 3, 1, 2)


def forward_fp8(q_codes, q_scales, k_codes, k_scales, vt_codes, v_scales, scale: float,
                causal: bool, heads=None, seqs=None, return_max: bool = False):
    """The FP8 forward's definition: exact fp64 attention over the dequantized
    inputs. Returns (o, lse) like ``attention_fp64.forward`` (dense layout;
    entries of heads or sequences outside the subset are NaN), and with
    ``return_max`` also the row maxima of the scaled scores [B, Hq, Sq].
    Dequantizes one (sequence, head) at a time, so a subset of a large problem
    stays small."""
    qc, kc, vc = np.asarray(q_codes), np.asarray(k_codes), np.asarray(vt_codes)
    qs, ks, vs = (np.asarray(x, dtype=np.float64) for x in (q_scales, k_scales, v_scales))
    B, Sq, Hq, d = qc.shape
    Sk, Hkv = kc.shape[1], kc.shape[2]
    group = Hq // Hkv
    o = np.full((B, Sq, Hq, d), np.nan)
    lse = np.full((B, Hq, Sq), np.nan)
    mx = np.full((B, Hq, Sq), np.nan)
    for b in range(B):
        if seqs is not None and b not in seqs:
            continue
        for h in (range(Hq) if heads is None else heads):
            g = h // group
            qh = e4m3_decode(qc[b, :, h]) * np.repeat(qs[b, h], BLOCK)[:Sq, None]
            kh = e4m3_decode(kc[b, :, g]) * np.repeat(ks[b, g], BLOCK)[:Sk, None]
            vh = e4m3_decode(vc[b, g, :, :Sk]).T * vs[b, g]
            o[b, :, h], lse[b, h], mx[b, h] = _attend_head(qh, kh, vh, scale, causal,
                                                           return_max=True)
    return (o, lse, mx) if return_max else (o, lse)
