"""Pins for the FP8 (e4m3) oracle: the format's fixed points, rounding, the
block quantizer and the FP8 forward's definition, each against something other
than the oracle's own formula (the format's defining constants, brute force,
invariants, and the fp64 attention oracle's own pins)."""
import numpy as np
import pytest

from oracle import attention_fp64 as A
from oracle import fp8_e4m3 as f8
from oracle import forward as fwd64


def test_format_fixed_points():
    # e4m3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities
    dec = f8.e4m3_decode
    assert dec(0x7E) == 448.0                       # largest finite: 1.75 * 2^8
    assert dec(0x08) == 2.0 ** -6                   # smallest normal
    assert dec(0x01) == 2.0 ** -9                   # smallest subnormal
    assert dec(0x07) == 7 * 2.0 ** -9               # largest subnormal
    assert dec(0x38) == 1.0                         # exponent field 7 = bias
    assert dec(0x00) == 0.0 and np.signbit(dec(0x80))
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    assert dec(0xFE) == -448.0
    # 254 finite codes (two NaN codes), 126 distinct positive nonzero values
    vals = dec(np.arange(256, dtype=np.uint8))
    finite = vals[np.isfinite(vals)]
    assert len(finite) == 254 and len(np.unique(finite[finite > 0])) == 126


def test_encode_exact_values_and_ties():
    enc = f8.e4m3_encode
    assert enc(1.0) == 0x38 and enc(448.0) == 0x7E and enc(-2.0 ** -9) == 0x81
    # 1 + 1/16 is halfway between 1 (mantissa 000) and 1.125 (001): even wins
    assert enc(1.0 + 1 / 16) == 0x38
    # 1 + 3/16 is halfway between 1.125 (001) and 1.25 (010): even wins
    assert enc(1.0 + 3 / 16) == 0x3A
    # just above a tie goes up
    assert enc(np.nextafter(1.0 + 1 / 16, 2.0)) == 0x39
    # subnormal ties: 2^-10 is halfway between 0 and 2^-9 -> 0 (even)
    assert enc(2.0 ** -10) == 0x00 and enc(3 * 2.0 ** -10) == 0x02
    # saturation (finite mode) and NaN
    assert enc(500.0) == 0x7E and enc(1e30) == 0x7E and enc(-1e30) == 0xFE
    assert enc(np.nan) == 0x7F


def test_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = f8.e4m3_encode(f8.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def test_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.uniform(-4, 2.7, 4000),
                        rng.uniform(-450, 450, 1000)]).astype(np.float32)
    codes = f8.e4m3_encode(x)
    table = f8.e4m3_decode(np.arange(256, dtype=np.uint8))
    ok = np.isfinite(table)
    for xi, ci in zip(x.astype(np.float64), codes):
        xs = np.clip(xi, -448.0, 448.0)
        dist = np.where(ok, np.abs(table - xs), np.inf)
        best = dist.min()
        assert dist[ci] == best                       # a nearest value
        ties = np.flatnonzero(dist == best)
        if len(np.unique(table[ties])) > 1:           # a true tie: the even code
            assert ci % 2 == 0


def test_encode_monotone():
    x = np.linspace(-460, 460, 200001)
    v = f8.e4m3_decode(f8.e4m3_encode(x))
    assert np.all(np.diff(v) >= 0)


def test_row_block_quantizer():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2, 300, 3, 64)) * rng.uniform(0.1, 5, (1, 300, 3, 1))).astype(np.float32)
    x[1, 128:256, 2] = 0.0                             # an all-zero block: scale 1, codes 0
    codes, scales = f8.quantize_row_blocks(x)
    assert scales.shape == (2, 3, 3)
    assert scales[1, 2, 1] == 1.0 and not codes[1, 128:256, 2].any()
    # the block maximum maps to 448 exactly (largest code), nothing exceeds it
    for b in range(2):
        for h in range(3):
            for i in range(3):
                blk = codes[b, i * 128:(i + 1) * 128, h]
                amax = np.abs(x[b, i * 128:(i + 1) * 128, h]).max()
                if amax > 0:
                    assert scales[b, h, i] == np.float32(amax / np.float32(448))
                if scales[b, h, i] != 1.0 or blk.any():
                    assert (blk & 0x7F).max() == 0x7E
    back = f8.dequantize_row_blocks(codes, scales)
    # relative error of every element within half an e4m3 step of its binade
    # (2^-4), or within half the subnormal step times the scale
    err = np.abs(back - x)
    rep = np.repeat(scales, 128, axis=2)[:, :, :300].transpose(0, 2, 1)[..., None]
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, rep * 2.0 ** -10) * (1 + 1e-6))


def test_v_quantizer_layout():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((2, 37, 2, 64)).astype(np.float32)
    codes, scales = f8.quantize_v_transposed(v)
    assert codes.shape == (2, 2, 64, 48) and not codes[..., 37:].any()
    for b in range(2):
        for h in range(2):
            assert scales[b, h] == np.float32(np.abs(v[b, :, h]).max() / np.float32(448))
            r = np.float32(1) / scales[b, h]
            assert r.dtype == np.float32 and (v[b, :, h] * r).dtype == np.float32
            assert np.array_equal(codes[b, h, :, :37].T, f8.e4m3_encode(v[b, :, h] * r))
    back = f8.dequantize_v_transposed(codes, scales, 37)
    assert np.abs(back - v).max() <= np.abs(v).max() * 2.0 ** -4


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_is_attention_of_dequantized_inputs(causal):
    """forward_fp8 equals the fp64 oracle on hand-dequantized inputs, and for
    inputs that are already e4m3 values times a power-of-two scale the
    quantize-dequantize round trip is the identity, so it equals the fp64
    oracle on the raw inputs."""
    rng = np.random.default_rng(5)
    B, S, H, d = 1, 200, 2, 64
    # inputs exactly representable: e4m3 values scaled by a power of two such
    # that each block's amax is exactly 448 * scale
    raw = f8.e4m3_decode(rng.integers(0, 0x7E, (B, S, H, d)).astype(np.uint8) | (rng.integers(0, 2, (B, S, H, d)) << 7).astype(np.uint8))
    raw = np.where(np.isnan(raw), 0.0, raw)
    raw[:, ::128, :, 0] = 448.0                       # pin every block's amax to 448
    x = (raw * 2.0 ** -6).astype(np.float32)
    qc, qs = f8.quantize_row_blocks(x)
    assert np.all(qs == np.float32(2.0 ** -6))
    assert np.array_equal(f8.dequantize_row_blocks(qc, qs), x.astype(np.float64))
    vc, vs = f8.quantize_v_transposed(x)
    o8, l8 = f8.forward_fp8(qc, qs, qc, qs, vc, vs, 0.125, causal)
    o, l = fwd64(x, x, x, 0.125, causal)
    assert np.allclose(o8, o, atol=1e-12) and np.allclose(l8, l, atol=1e-12)
    # the row maxima it returns on request are the fp64 oracle's
    _, _, m8 = f8.forward_fp8(qc, qs, qc, qs, vc, vs, 0.125, causal, return_max=True)
    for h in range(H):
        xh = x[0, :, h]
        _, _, mh = A.attend_head(xh, xh, xh, 0.125, causal, return_max=True)
        assert np.allclose(m8[0, h], mh, atol=1e-12)


@pytest.mark.parametrize("Sk", [128, 2048])
def test_weight_rounding_error_matches_the_tolerance_derivation(Sk):
    """The FP8 forward's O tolerance (rel-L2 5e-2) comes from rounding each
    softmax weight to e4m3 (relative error <= 2^-4, RMS <= 2^-4/sqrt(3) = 3.6%).
    Rounding exact weights (as 2^7 p, the kernel's storage) with the oracle's
    codec on random rows gives an output error of that size: below the bound,
    and not so far below that the bound would be vacuous."""
    rng = np.random.default_rng(Sk)
    rows, d = 256, 64
    s = rng.standard_normal((rows, Sk))                  # scores ~ N(0, 1)
    v = rng.standard_normal((Sk, d))
    p = np.exp2((s - s.max(axis=1, keepdims=True)) * 1.4426950408889634 + 7)
    o = (p @ v) / p.sum(axis=1, keepdims=True)
    p8 = f8.e4m3_decode(f8.e4m3_encode(p))
    o8 = (p8 @ v) / p.sum(axis=1, keepdims=True)         # row sum from the fp32 weights
    rel = np.linalg.norm(o8 - o) / np.linalg.norm(o)
    assert 0.005 < rel < 0.05
    assert np.abs(p8 / np.where(p > 0, p, 1) - 1)[p >= 2.0 ** -6].max() <= 2.0 ** -4
    # Element-wise: a weight in e4m3's normal range is off by at most 2^-4 of
    # itself, one below it (stored value < 2^-6) by at most half the smallest
    # subnormal step, 2^-10; divided by the row sum l >= 2^7 (the row maximum
    # is stored as 2^7), each output element is off by at most
    # 2^-4 * sum_j p_j |v_jc| / l + 2^-10 * sum_j |v_jc| / l.
    l = p.sum(axis=1, keepdims=True)
    bound = 2.0 ** -4 * (p @ np.abs(v)) / l + 2.0 ** -10 * np.abs(v).sum(axis=0) / l
    err = np.abs(o8 - o)
    assert np.all(err <= bound)
    # not vacuous: independent rounding errors partly cancel over many keys,
    # so the worst case is approached less closely as Sk grows
    assert (err / bound).max() > 0.05


# ---------------------------------------------------------------------------
# Mutation tests: plant a plausible mistake in a copy of the FP8 oracle and
# check that at least one pin catches it.
# ---------------------------------------------------------------------------
import inspect  # noqa: E402

_F8_MUTATIONS = [
    ("np.exp2(e.astype(np.float64) - 7)", "np.exp2(e.astype(np.float64) - 8)"),   # exponent bias
    ("(hi % 2 == 0)", "(hi % 2 == 1)"),                                            # ties to odd
    ("amax / np.float32(E4M3_MAX)", "amax / np.float32(447)"),                     # scale constant
    ("e4m3_encode(blk * (np.float32(1) / s)).T", "e4m3_encode(blk * (np.float32(1) / s)).T[::-1]"),  # V^T rows
    ("vh = e4m3_decode(vc[b, g, :, :Sk]).T * vs[b, g]", "vh = e4m3_decode(vc[b, g, :, :Sk]).T"),  # V scale
    ("g = h // group", "g = h % Hkv"),                                             # GQA head map
    ("np.repeat(qs[b, h], BLOCK)[:Sq, None]", "qs[b, h, 0]"),                      # one Q scale
]


def _f8_mutant(old, new):
    src = inspect.getsource(f8)
    assert old in src, old
    src = src.replace(old, new).replace(
        "from .attention_fp64 import attend_head as _attend_head",
        "from oracle.attention_fp64 import attend_head as _attend_head")
    ns = {"__name__": "fp8_mutant"}
    exec(compile(src, "<fp8_mutant>", "exec"), ns)
    return ns


def _f8_pins_pass(m):
    try:
        dec, enc = m["e4m3_decode"], m["e4m3_encode"]
        if not (dec(0x7E) == 448.0 and dec(0x08) == 2.0 ** -6 and dec(0x01) == 2.0 ** -9
                and dec(0x38) == 1.0):
            return False
        if not (enc(1.0 + 1 / 16) == 0x38 and enc(1.0 + 3 / 16) == 0x3A and enc(2.0 ** -10) == 0):
            return False
        codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
        if not np.array_equal(enc(dec(codes)), codes):
            return False
        rng = np.random.default_rng(11)
        x = rng.standard_normal((1, 300, 4, 64)).astype(np.float32) * rng.uniform(
            0.2, 3, (1, 300, 1, 1)).astype(np.float32)
        qc, qs = m["quantize_row_blocks"](x)
        for i in range(3):
            amax = np.abs(x[0, i * 128:(i + 1) * 128, 1]).max()
            if qs[0, 1, i] != np.float32(amax / np.float32(448)):
                return False
        vc, vs = m["quantize_v_transposed"](x[:, :, :2])
        r = np.float32(1) / vs[0, 1]
        if not np.array_equal(vc[0, 1, :, :300].T, f8.e4m3_encode(x[0, :, 1] * r)):
            return False
        # varying block scales and GQA: forward_fp8 against fp64 attention over
        # the dequantized inputs, built with the pinned dequantizers
        kc, ks = m["quantize_row_blocks"](x[:, :, :2])
        for causal in (False, True):
            o8, l8 = m["forward_fp8"](qc, qs, kc, ks, vc, vs, 0.125, causal)
            q = f8.dequantize_row_blocks(qc, qs)
            k = f8.dequantize_row_blocks(kc, ks)
            v = f8.dequantize_v_transposed(vc, vs, 300)
            o, l = fwd64(q, k, v, 0.125, causal)
            if not (np.allclose(o8, o, atol=1e-12) and np.allclose(l8, l, atol=1e-12)):
                return False
    except Exception:
        return False
    return True


@pytest.mark.parametrize("old,new", _F8_MUTATIONS, ids=[m[1][:28] for m in _F8_MUTATIONS])
def test_fp8_pins_catch_planted_mistakes(old, new):
    assert _f8_pins_pass(_f8_mutant("", ""))          # the unmodified copy passes
    assert not _f8_pins_pass(_f8_mutant(old, new))
