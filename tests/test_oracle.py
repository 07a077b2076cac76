"""Pins for the fp64 oracle: checks against what the mathematics fixes.

None of these re-types the oracle's formula: they use hand-derived closed forms,
invariants, a pure-Python brute force, torch's fp64 SDPA (a library special
case), central finite differences, structural equivalences, and mutation tests
that plant mistakes in a copy of the oracle and require a pin to catch them.
"""
import inspect
import json
import math
import os
import textwrap

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_fp64 as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _ev(x):
    if isinstance(x, list):
        return [_ev(y) for y in x]
    return float(eval(x, {"__builtins__": {}}, {"e": math.e, "ln": math.log, "inf": math.inf}))


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_golden_closed_forms(case):
    q, k, v = (np.array(_ev(case[n])) for n in ("q", "k", "v"))
    scale = _ev(case["scale"])
    o, lse = oracle.attend_head(q, k, v, scale, case["causal"])
    np.testing.assert_allclose(o, np.array(_ev(case["o"])), rtol=0, atol=1e-14)
    want = np.array(_ev(case["lse"]))
    assert np.array_equal(np.isinf(lse), np.isinf(want))
    np.testing.assert_allclose(lse[np.isfinite(want)], want[np.isfinite(want)], atol=1e-14)
    if "do" in case:
        do = np.array(_ev(case["do"]))
        dq, dk, dv = oracle.attend_head_backward(q, k, v, do, scale, case["causal"])
        np.testing.assert_allclose(dq, np.array(_ev(case["dq"])), atol=1e-14)
        np.testing.assert_allclose(dk, np.array(_ev(case["dk"])), atol=1e-14)
        np.testing.assert_allclose(dv, np.array(_ev(case["dv"])), atol=1e-14)


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(7, 7), (5, 9), (9, 5), (130, 300)])
def test_rows_sum_to_one(causal, nq, nk):
    """exp(S - LSE) is a probability distribution over the visible keys of each row."""
    q, k, v = _rand((nq, 8), 1), _rand((nk, 8), 2), _rand((nk, 8), 3)
    scale = 0.37
    _, lse = oracle.attend_head(q, k, v, scale, causal)
    s = scale * q @ k.T
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    vis = (j <= i + nk - nq) if causal else np.ones_like(s, dtype=bool)
    rows = vis.any(axis=1)
    p = np.where(vis, np.exp(s - np.where(rows, lse, 0)[:, None]), 0.0)
    np.testing.assert_allclose(p.sum(axis=1)[rows], 1.0, atol=1e-13)
    assert np.all(np.isinf(lse[~rows]))


@pytest.mark.parametrize("causal", [False, True])
def test_v_all_ones_gives_ones(causal):
    q, k = _rand((40, 16), 4, 3.0), _rand((40, 16), 5, 3.0)
    o, _ = oracle.attend_head(q, k, np.ones((40, 16)), 0.25, causal)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


def test_causal_row0_is_v0():
    q, k, v = _rand((33, 8), 6), _rand((33, 8), 7), _rand((33, 8), 8)
    o, lse = oracle.attend_head(q, k, v, 0.5, True)
    np.testing.assert_array_equal(o[0], v[0])
    assert lse[0] == pytest.approx(0.5 * q[0] @ k[0], abs=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(16, 16), (6, 11)])
def test_zero_queries_closed_form(causal, nq, nk):
    """Q = 0: uniform softmax over the visible keys; LSE = ln(#visible)."""
    v = _rand((nk, 4), 9)
    o, lse = oracle.attend_head(np.zeros((nq, 4)), _rand((nk, 4), 10), v, 1.0, causal)
    for i in range(nq):
        n = min(nk, i + 1 + nk - nq) if causal else nk
        assert lse[i] == pytest.approx(math.log(n), abs=1e-14)
        np.testing.assert_allclose(o[i], v[:n].mean(axis=0), atol=1e-14)


def _brute_force(q, k, v, scale, causal):
    """Pure-Python loops with math.exp: one row at a time, no numpy arithmetic."""
    nq, nk, dv = len(q), len(k), len(v[0])
    out, lses, maxes = [], [], []
    for i in range(nq):
        scores = []
        for j in range(nk):
            if causal and j > i + nk - nq:
                continue
            scores.append((j, scale * sum(a * b for a, b in zip(q[i], k[j]))))
        mx = max(s for _, s in scores)
        w = [(j, math.exp(s - mx)) for j, s in scores]
        tot = sum(x for _, x in w)
        out.append([sum(x * v[j][c] for j, x in w) / tot for c in range(dv)])
        lses.append(mx + math.log(tot))
        maxes.append(mx)
    return np.array(out), np.array(lses), np.array(maxes)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,d", [(5, 5, 3), (3, 6, 2), (4, 4, 1)])
def test_brute_force_tiny(causal, nq, nk, d):
    q, k, v = _rand((nq, d), 11, 2), _rand((nk, d), 12, 2), _rand((nk, d + 1), 13)
    o, lse, m = oracle.attend_head(q, k, v, 0.7, causal, return_max=True)
    ob, lb, mb = _brute_force(q.tolist(), k.tolist(), v.tolist(), 0.7, causal)
    np.testing.assert_allclose(o, ob, atol=1e-13)
    np.testing.assert_allclose(lse, lb, atol=1e-13)
    np.testing.assert_allclose(m, mb, atol=1e-13)
    o2, lse2 = oracle.attend_head(q, k, v, 0.7, causal)      # the flag changes nothing else
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_fp64_fwd_bwd(causal):
    """Library special case: torch's fp64 SDPA (Sq == Sk, so causal alignments agree) + autograd."""
    B, S, H, d = 2, 37, 3, 8
    q, k, v, do = (_rand((B, S, H, d), 20 + i) for i in range(4))
    scale = 0.3
    tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3), requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do.transpose(0, 2, 1, 3)))
    o, _ = oracle.forward(q, k, v, scale, causal)
    np.testing.assert_allclose(o, to.detach().numpy().transpose(0, 2, 1, 3), atol=1e-12)
    dq, dk, dv = oracle.backward(q, k, v, do, scale, causal)
    for mine, ref in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(mine, ref.grad.numpy().transpose(0, 2, 1, 3), atol=1e-11)


def _loss(q, k, v, do, scale, causal):
    o, _ = oracle.attend_head(q, k, v, scale, causal)
    return float((o * do).sum())


@pytest.mark.parametrize("causal,nq,nk", [(False, 5, 7), (True, 6, 6), (True, 4, 7)])
def test_backward_finite_differences(causal, nq, nk):
    d, scale, h = 4, 0.6, 1e-6
    q, k, v, do = _rand((nq, d), 30), _rand((nk, d), 31), _rand((nk, d), 32), _rand((nq, d), 33)
    dq, dk, dv = oracle.attend_head_backward(q, k, v, do, scale, causal)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, do, scale, causal)
            x[idx] = old - h
            lm = _loss(q, k, v, do, scale, causal)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_backward_finite_differences_gqa_varlen():
    """Whole-batch backward: GQA group sums and packed sequences, against finite differences."""
    lengths, hq, hkv, d, scale, h = [3, 5], 4, 2, 3, 0.5, 1e-6
    T = sum(lengths)
    cu = np.array([0, 3, 8])
    q, k, v, do = _rand((T, hq, d), 40), _rand((T, hkv, d), 41), _rand((T, hkv, d), 42), _rand((T, hq, d), 43)
    dq, dk, dv = oracle.backward(q, k, v, do, scale, True, cu_seqlens=cu)

    def loss():
        o, _ = oracle.forward(q, k, v, scale, True, cu_seqlens=cu)
        return float((o * do).sum())

    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss()
            x[idx] = old - h
            lm = loss()
            x[idx] = old
            assert g[idx] == pytest.approx((lp - lm) / (2 * h), rel=1e-6, abs=1e-8)


def test_separate_key_boundaries_uniform_scores():
    """Packed layout with separate query/key boundaries, scale 0: every visible
    key gets the same weight, so row i of a sequence with q_len queries and
    k_len keys is the plain mean of V over its first i + k_len - q_len + 1 keys
    (bottom-right causal) or over all keys, and LSE = ln(number of keys)."""
    cu_q, cu_k = np.array([0, 3, 4, 9]), np.array([0, 5, 5, 8])   # k_len 5, 0, 3
    hq, hkv, d = 2, 1, 3
    q, k, v = _rand((9, hq, d), 60), _rand((8, hkv, d), 61), _rand((8, hkv, d), 62)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, 0.0, causal, cu_seqlens=cu_q, cu_seqlens_k=cu_k)
        for s in range(3):
            ql, kl = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
            for i in range(ql):
                n = kl if not causal else max(0, min(kl, i + kl - ql + 1))
                row = cu_q[s] + i
                for h in range(hq):
                    if n == 0:
                        assert np.all(o[row, h] == 0) and lse[h, row] == np.inf
                    else:
                        want = v[cu_k[s]:cu_k[s] + n, 0].mean(axis=0)
                        np.testing.assert_allclose(o[row, h], want, atol=1e-14)
                        assert lse[h, row] == pytest.approx(np.log(n), abs=1e-14)


def test_separate_key_boundaries_finite_differences():
    """Backward with separate boundaries (prefill over cached keys: more keys than
    queries, and one sequence with fewer), against central finite differences."""
    cu_q, cu_k = np.array([0, 2, 5]), np.array([0, 4, 6])
    hq, hkv, d, scale, h = 2, 1, 3, 0.5, 1e-6
    q, k, v, do = _rand((5, hq, d), 70), _rand((6, hkv, d), 71), _rand((6, hkv, d), 72), _rand((5, hq, d), 73)
    dq, dk, dv = oracle.backward(q, k, v, do, scale, True, cu_seqlens=cu_q, cu_seqlens_k=cu_k)

    def loss():
        o, _ = oracle.forward(q, k, v, scale, True, cu_seqlens=cu_q, cu_seqlens_k=cu_k)
        return float((o * do).sum())

    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss()
            x[idx] = old - h
            lm = loss()
            x[idx] = old
            assert g[idx] == pytest.approx((lp - lm) / (2 * h), rel=1e-6, abs=1e-8)


def test_gqa_equals_mha_with_repeated_kv():
    B, S, hq, hkv, d = 2, 19, 6, 2, 5
    q, k, v, do = _rand((B, S, hq, d), 50), _rand((B, S, hkv, d), 51), _rand((B, S, hkv, d), 52), _rand((B, S, hq, d), 53)
    kr, vr = np.repeat(k, hq // hkv, axis=2), np.repeat(v, hq // hkv, axis=2)
    o1, l1 = oracle.forward(q, k, v, 0.4, True)
    o2, l2 = oracle.forward(q, kr, vr, 0.4, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    dq1, dk1, dv1 = oracle.backward(q, k, v, do, 0.4, True)
    dq2, dk2, dv2 = oracle.backward(q, kr, vr, do, 0.4, True)
    np.testing.assert_allclose(dq1, dq2, atol=1e-14)
    np.testing.assert_allclose(dk1, dk2.reshape(B, S, hkv, hq // hkv, d).sum(axis=3), atol=1e-13)
    np.testing.assert_allclose(dv1, dv2.reshape(B, S, hkv, hq // hkv, d).sum(axis=3), atol=1e-13)


def test_varlen_equals_per_sequence_dense():
    lengths, H, d = [4, 1, 9, 6], 2, 3
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T = cu[-1]
    q, k, v, do = (_rand((T, H, d), 60 + i) for i in range(4))
    o, lse = oracle.forward(q, k, v, 0.8, True, cu_seqlens=cu)
    dq, dk, dv = oracle.backward(q, k, v, do, 0.8, True, cu_seqlens=cu)
    for i, L in enumerate(lengths):
        sl = slice(cu[i], cu[i + 1])
        od, ld = oracle.forward(q[None, sl], k[None, sl], v[None, sl], 0.8, True)
        np.testing.assert_array_equal(o[sl], od[0])
        np.testing.assert_array_equal(lse[:, sl], ld[0])
        g = oracle.backward(q[None, sl], k[None, sl], v[None, sl], do[None, sl], 0.8, True)
        for a, b in zip((dq, dk, dv), g):
            np.testing.assert_array_equal(a[sl], b[0])


def test_row_chunking_is_invisible():
    q, k, v, do = _rand((50, 4), 70), _rand((50, 4), 71), _rand((50, 4), 72), _rand((50, 4), 73)
    a = oracle.attend_head_backward(q, k, v, do, 0.5, True, row_chunk=7)
    b = oracle.attend_head_backward(q, k, v, do, 0.5, True, row_chunk=1000)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-14)


@pytest.mark.parametrize("tau", [0.0, 1.0, 2.0, 8.0])
@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_equals_naive(tau, causal):
    q, k, v = _rand((97, 16), 80, 2.0), _rand((300, 16), 81, 2.0), _rand((300, 16), 82)
    on, ln_ = oracle.online_attend_head(q, k, v, 0.5, causal, block_n=32, tau=tau)
    o, lse = oracle.attend_head(q, k, v, 0.5, causal)
    np.testing.assert_allclose(on, o, atol=1e-12)
    np.testing.assert_allclose(ln_, lse, atol=1e-12)


def test_conditional_rescale_skips_work():
    q, k, v = _rand((64, 16), 83, 2.0), _rand((1024, 16), 84, 2.0), _rand((1024, 16), 85)
    counts = [oracle.online_attend_head(q, k, v, 0.5, False, 64, tau, True)[2] for tau in (0.0, 2.0, 8.0)]
    assert counts[0] > counts[1] > counts[2]


def test_exp2_method_degree3_bound():
    """The range-reduced degree-3 method reaches relative error < 2^-13 on [-126, 0]."""
    c = oracle.fit_exp2_poly(3)
    assert c[0] == 1.0
    bf16 = np.arange(0x8000, 0x10000, dtype=np.uint32) << 16        # every negative bf16
    with np.errstate(invalid="ignore"):
        xb = bf16.view(np.float32).astype(np.float64)
    xs = np.concatenate([xb[np.isfinite(xb) & (xb >= -126)], np.linspace(-126, 0, 400001), [0.0]])
    rel = np.abs(oracle.exp2_range_reduced(xs, c) / oracle.exp2_exact(xs) - 1)
    assert rel.max() < 2.0 ** -13
    assert oracle.exp2_range_reduced(0.0, c) == 1.0
    # lower degrees do not meet the bound (the pin is sensitive to the method's degree)
    rel2 = np.abs(oracle.exp2_range_reduced(xs, oracle.fit_exp2_poly(2)) / oracle.exp2_exact(xs) - 1)
    assert rel2.max() > 2.0 ** -13


# ---------------------------------------------------------------------------
# Mutation tests: plant a plausible mistake in a copy of the oracle and check
# that at least one pin above catches it.
# ---------------------------------------------------------------------------
_MUTATIONS = [
    ("(nk - nq)", "(nq - nk)"),          # wrong causal alignment
    ("j <= i", "j < i"),                # off-by-one causal mask
    ("s = scale * (q[r0:r1] @ k.T)", "s = (q[r0:r1] @ k.T)"),   # dropped scale
    ("np.exp(s - m_safe[:, None])", "np.exp(s + m_safe[:, None])"),  # wrong sign
    ("m_safe + np.log", "m_safe - np.log"),   # wrong LSE sign
    ("(p @ v)", "(p @ v[::-1])"),        # wrong V row index
]


def _mutant(src_old, src_new):
    src = textwrap.dedent(inspect.getsource(A))
    assert src_old in src, src_old
    mod_src = src.replace(src_old, src_new)
    ns = {"__name__": "mutant"}
    exec(compile(mod_src, "<mutant>", "exec"), ns)
    return ns


def _pins_pass(ns):
    attend = ns["attend_head"]
    try:
        for case in _cases():
            q, k, v = (np.array(_ev(case[n])) for n in ("q", "k", "v"))
            o, lse = attend(q, k, v, _ev(case["scale"]), case["causal"])
            want = np.array(_ev(case["lse"]))
            if not np.allclose(o, np.array(_ev(case["o"])), atol=1e-12):
                return False
            if not np.array_equal(np.isinf(lse), np.isinf(want)):
                return False
            if not np.allclose(lse[np.isfinite(want)], want[np.isfinite(want)], atol=1e-12):
                return False
        for causal in (False, True):
            q, k, v = _rand((5, 3), 11, 2), _rand((6, 3), 12, 2), _rand((6, 4), 13)
            o, lse = attend(q, k, v, 0.7, causal)
            ob, lb, _ = _brute_force(q.tolist(), k.tolist(), v.tolist(), 0.7, causal)
            if not (np.allclose(o, ob, atol=1e-12) and np.allclose(lse, lb, atol=1e-12)):
                return False
    except Exception:
        return False
    return True


@pytest.mark.parametrize("old,new", _MUTATIONS, ids=[m[1][:24] for m in _MUTATIONS])
def test_pins_catch_planted_mistakes(old, new):
    assert _pins_pass(_mutant("", ""))          # the unmodified copy passes
    assert not _pins_pass(_mutant(old, new))
