"""The LPT work scheduler, run on the host through the C ABI (no GPU).

Costs are recomputed here by brute force from the masking rule (count the inner
blocks that hold at least one key visible to at least one row of the unit), so
the test does not share the scheduler's closed forms.
"""
import itertools

import pytest

from fa_testing_lib import fa_sched_list


def _seqs(B, cu, Sq, Sk):
    if cu is None:
        return [(Sq, Sk)] * B
    return [(cu[i + 1] - cu[i],) * 2 for i in range(len(cu) - 1)]


def _visible(i, j, ql, kl, causal):
    return j < kl and i < ql and (not causal or j <= i + kl - ql)


# kind -> (query-unit rows or key-unit rows, inner block rows, units over queries?)
_KINDS = {0: (256, 128, True), 1: (128, 64, False), 2: (128, 128, False), 3: (128, 128, True),
          4: (256, 128, False), 5: (128, 64, True)}


def _brute_units(kind, B, cu, Sq, Sk, heads, causal):
    U, I, over_queries = _KINDS[kind]
    units = {}
    for s, (ql, kl) in enumerate(_seqs(B, cu, Sq, Sk)):
        if over_queries:
            for m in range((ql + U - 1) // U):
                rows = range(m * U, min(ql, m * U + U))
                # KV blocks walked: from block 0 up to the last block with a visible key
                last = -1
                for jb in range((kl + I - 1) // I):
                    if any(_visible(i, j, ql, kl, causal) for i in (rows[-1],)
                           for j in range(jb * I, min(kl, jb * I + I))):
                        last = jb
                for h in range(heads):
                    units[(s, m, h)] = last + 1
        else:
            for n in range((kl + U - 1) // U):
                keys = range(n * U, min(kl, n * U + U))
                first = None
                for ib in range((ql + I - 1) // I):
                    if any(_visible(i, keys[0], ql, kl, causal) for i in range(ib * I, min(ql, ib * I + I))):
                        first = ib
                        break
                c = 0 if first is None else (ql + I - 1) // I - first
                for h in range(heads):
                    units[(s, n, h)] = c
    return units


CASES = [
    (0, 2, None, 600, 600, 3, True), (0, 2, None, 600, 600, 3, False), (0, 3, None, 1, 1, 2, True),
    (0, 1, None, 300, 1000, 2, True), (0, 1, None, 1000, 300, 2, True),
    (0, 4, [0, 1, 1, 700, 3000], 3000, 3000, 2, True), (0, 3, [0, 129, 385, 1000], 1000, 1000, 4, False),
    (1, 2, None, 600, 600, 3, True), (1, 2, None, 600, 600, 3, False), (1, 1, None, 300, 1000, 2, True),
    (1, 1, None, 1000, 300, 2, True), (1, 4, [0, 1, 1, 700, 3000], 3000, 3000, 2, True),
    (2, 2, None, 600, 600, 3, True), (2, 2, None, 600, 600, 3, False), (2, 1, None, 300, 1000, 2, True),
    (2, 1, None, 1000, 300, 2, True), (2, 4, [0, 1, 1, 700, 3000], 3000, 3000, 2, True),
    (3, 2, None, 600, 600, 3, True), (3, 2, None, 600, 600, 3, False), (3, 1, None, 300, 1000, 2, True),
    (3, 1, None, 1000, 300, 2, True), (3, 3, [0, 129, 385, 1000], 1000, 1000, 4, True),
    (4, 2, None, 600, 600, 3, True), (4, 1, None, 300, 1000, 2, True), (4, 1, None, 1000, 300, 2, True),
    (4, 4, [0, 1, 1, 700, 3000], 3000, 3000, 2, True),
    (5, 2, None, 600, 600, 3, True), (5, 2, None, 600, 600, 3, False), (5, 1, None, 300, 1000, 2, True),
    (5, 1, None, 1000, 300, 2, True), (5, 3, [0, 129, 385, 1000], 1000, 1000, 4, True),
]


@pytest.mark.parametrize("hpg", [0, 1, 2])
@pytest.mark.parametrize("grid", [1, 5, 152])
@pytest.mark.parametrize("case", CASES)
def test_every_unit_once_with_its_cost(case, grid, hpg):
    kind, B, cu, Sq, Sk, heads, causal = case
    want = _brute_units(kind, B, cu, Sq, Sk, heads, causal)
    got = {}
    for cta in range(grid):
        for (s, m, h, c) in fa_sched_list(kind, B, cu, Sq, Sk, heads, causal, grid, cta, hpg):
            assert (s, m, h) not in got
            got[(s, m, h)] = c
    assert got == want


@pytest.mark.parametrize("hpg", [0, 1, 2, 3])
@pytest.mark.parametrize("case", CASES)
def test_list_order_is_grouped_then_longest_first(case, hpg):
    """Interleaving the CTAs' lists back into list order gives head groups in
    order, each in non-increasing cost (pure LPT when one group holds all heads)."""
    kind, B, cu, Sq, Sk, heads, causal = case
    G = 7
    per = [fa_sched_list(kind, B, cu, Sq, Sk, heads, causal, G, b, hpg) for b in range(G)]
    order = []
    for k in itertools.count():
        row = [per[b][k] if k < len(per[b]) else None for b in range(G)]
        if all(x is None for x in row):
            break
        if k % 2:
            row = row[::-1]
        order += [x for x in row if x is not None]
    if hpg == 0:
        return   # group size chosen from the grid; covered by the other values
    groups = [u[2] // hpg for u in order]
    assert groups == sorted(groups)
    for g in set(groups):
        costs = [u[3] for u in order if u[2] // hpg == g]
        assert costs == sorted(costs, reverse=True)


def test_auto_group_covers_the_grid():
    """The kernels' own group size: the fewest heads whose units fill the grid."""
    units = fa_sched_list(1, 1, None, 32768, 32768, 32, True, 152, 0)
    assert len({u[2] for u in units[:1]}) == 1
    # 256 key blocks per head >= 152 CTAs: one head per group, so CTA 0's first
    # two units come from heads 0 and 0 or 1, never from far-apart heads
    assert units[0][2] == 0 and units[1][2] <= 1


def test_causal_balance_near_lpt_bound():
    """Long causal batch: per-CTA total cost within a few percent of the mean."""
    G = 152
    # the kernels' choices: forward and dQ pass one group, dK/dV pass and one-pass auto
    for kind, hpg in ((0, 32), (1, 0), (2, 0), (3, 32), (4, 0)):
        g = G // 2 if kind == 4 else G           # the pair kernel's grid counts CTA pairs
        loads = [sum(u[3] for u in fa_sched_list(kind, 1, None, 32768, 32768, 32, True, g, b, hpg))
                 for b in range(g)]
        mean = sum(loads) / g
        assert max(loads) <= 1.03 * mean, (kind, max(loads) / mean)


def _graham(costs, G):
    """Graham's list scheduling of the costs in LPT order: each next unit goes
    to the least-loaded of G workers; returns the largest load."""
    import heapq
    loads = [0] * G
    for c in sorted(costs, reverse=True):
        heapq.heapreplace(loads, loads[0] + c)
    return max(loads)


def test_varlen_balance_near_lpt_bound():
    """The packed causal workload (16 sequences, lengths log-uniform on
    [128, 16384] drawn from seed 4, 32 heads) on 152 CTAs: the static snake
    deal of the LPT list keeps every CTA's total cost within 5% of the mean,
    and within 1% of what Graham's greedy list scheduling reaches, for the
    forward, the dK/dV pass, the dQ pass and the pair dK/dV pass, each with
    the head grouping its kernel uses for packed layouts (one group)."""
    import torch
    from attn_inputs import WORKLOADS, varlen_lengths
    w = WORKLOADS["varlen16_causal"]
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    lengths = varlen_lengths(gen, w.varlen_nseq, w.varlen_lo, w.varlen_hi)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    T = cu[-1]
    for kind in (0, 2, 3, 4):
        G = 76 if kind == 4 else 152               # the pair kernel's grid counts CTA pairs
        per = [fa_sched_list(kind, len(lengths), cu, T, T, w.Hq, True, G, b, w.Hq)
               for b in range(G)]
        loads = [sum(u[3] for u in units) for units in per]
        mean = sum(loads) / G
        assert max(loads) <= 1.05 * mean, (kind, max(loads) / mean)
        greedy = _graham([u[3] for units in per for u in units], G)
        assert max(loads) <= 1.01 * greedy, (kind, max(loads) / greedy)


def test_short_causal_balance_matches_greedy():
    """The short causal workload (B=4, H=16, S=2048) on 152 CTAs, each kernel
    with the head grouping it uses there (one group: the K/V and Q/dO of all
    heads fit L2): the static snake deal's largest per-CTA cost equals that of
    Graham's greedy list scheduling. For the forward that is 32 blocks, the
    optimum: every unit costs an even number of blocks and the mean is 30.3."""
    G = 152
    for kind in (0, 2, 3):
        per = [fa_sched_list(kind, 4, None, 2048, 2048, 16, True, G, b, 16) for b in range(G)]
        loads = [sum(u[3] for u in units) for units in per]
        costs = [u[3] for units in per for u in units]
        assert len(costs) == (512 if kind == 0 else 1024)
        assert max(loads) == _graham(costs, G), kind
        if kind == 0:
            assert all(c % 2 == 0 for c in costs) and max(loads) == 32
