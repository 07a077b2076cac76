"""Context-parallel ring (exact_attention_smem_gb300.ring) on the CPU.

The ring's schedule is checked on its own (every visible (query chunk, key
chunk) pair exactly once, zigzag chunks balance causal work), and the whole
exchange runs on 2 and 3 gloo ranks with the fp64 oracle as the per-pair
forward: each rank's merged output must equal the oracle's attention over the
full sequence at that rank's rows. The backward exchange runs the same way,
with an fp64 per-pair backward written here from the gradient formulas (given
the merged O and LSE); each rank's dQ, dK, dV must equal the oracle's
backward over the full sequence at its chunks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from exact_attention_smem_gb300 import ring


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
@pytest.mark.parametrize("world", [1, 2, 3, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_schedule_covers_every_visible_pair_once(world, layout, causal):
    n = ring.num_chunks(world, layout)
    seen = {}
    for rank in range(world):
        mine = ring.chunk_ids(world, rank, layout)
        steps = ring.ring_schedule(world, rank, causal, layout)
        assert [src for src, _ in steps] == [(rank - s) % world for s in range(world)]
        for src, pairs in steps:
            theirs = ring.chunk_ids(world, src, layout)
            for qi, ki, m in pairs:
                key = (mine[qi], theirs[ki])
                assert key not in seen
                seen[key] = m
    want = {}
    for a in range(n):
        for b in range(n):
            if not causal or b < a:
                want[(a, b)] = "full"
            elif b == a:
                want[(a, b)] = "causal"
    assert seen == want


@pytest.mark.parametrize("world", [2, 3, 4, 8])
def test_zigzag_balances_causal_work(world):
    """Causal work per rank (a full pair = 1, a diagonal pair = 1/2) is equal
    under the zigzag layout; under the contiguous layout rank r does r + 1/2."""
    def work(layout):
        return [sum(1.0 if m == "full" else 0.5
                    for _, pairs in ring.ring_schedule(world, r, True, layout) for _, _, m in pairs)
                for r in range(world)]
    z = work("zigzag")
    assert max(z) == min(z)
    c = work("contiguous")
    assert c == [r + 0.5 for r in range(world)]          # r full pairs + the diagonal


def _oracle_attend(q, k, v, causal, scale, out, lse):
    import oracle
    o, l = oracle.forward(q, k, v, scale, causal)
    out.copy_(torch.from_numpy(o))
    lse.copy_(torch.from_numpy(l))


def _lse_merge(o_parts, lse_parts):
    """Log-sum-exp combination of the parts (test side)."""
    lse = torch.logsumexp(lse_parts, dim=0)                     # [B, H, S]
    w = torch.exp(lse_parts - lse)                              # [P, B, H, S]
    o = (w.permute(0, 1, 3, 2)[..., None] * o_parts).sum(0)     # [B, S, H, d]
    return o, lse


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    errs = []
    try:
        for layout in ("zigzag", "contiguous"):
            for causal in (True, False):
                g = torch.Generator().manual_seed(17 + world)
                B, S, Hq, Hkv, d = 2, 48, 4, 2, 8
                qf = torch.randn(B, S, Hq, d, generator=g, dtype=torch.float64)
                kf = torch.randn(B, S, Hkv, d, generator=g, dtype=torch.float64)
                vf = torch.randn(B, S, Hkv, d, generator=g, dtype=torch.float64)
                scale = 0.3
                qs, ks, vs = (ring.split_sequence(t, world, rank, layout) for t in (qf, kf, vf))
                out = ring.ring_forward(qs, ks, vs, causal, scale, layout=layout,
                                        attend=_oracle_attend, merge=_lse_merge)
                ro, rl = oracle.forward(qf, kf, vf, scale, causal)
                c = S // ring.num_chunks(world, layout)
                for (o, lse), a in zip(out, ring.chunk_ids(world, rank, layout)):
                    rows = slice(a * c, (a + 1) * c)
                    errs.append(float(np.abs(o.numpy() - ro[:, rows]).max()))
                    errs.append(float(np.abs(lse.numpy() - rl[:, :, rows]).max()))
        q.put((rank, max(errs)))
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_on_gloo_ranks_equals_full_attention(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _ in res] == list(range(world))
    for _, err in res:
        assert err <= 1e-12


def _pair_backward(q, k, v, o, lse, do, causal, scale, dq, dk, dv):
    """fp64 gradient terms of one (query chunk, key chunk) pair, with the
    query rows' LSE and O over all keys: P = exp(S - LSE), D = rowsum(dO * O),
    dS = P (dP - D); dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO (test side)."""
    B, Sq, Hq, d = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    kk, vv = k.repeat_interleave(g, dim=2), v.repeat_interleave(g, dim=2)
    s = torch.einsum("bqhd,bkhd->bhqk", q, kk) * scale
    if causal:
        hide = torch.ones(Sq, Sk, dtype=torch.bool).triu(Sk - Sq + 1)
        s = s.masked_fill(hide, float("-inf"))
    p = torch.exp(s - lse[..., None])
    dp = torch.einsum("bqhd,bkhd->bhqk", do, vv)
    D = (do * o).sum(-1).permute(0, 2, 1)
    ds = p * (dp - D[..., None])
    dq.copy_(torch.einsum("bhqk,bkhd->bqhd", ds, kk) * scale)
    dk.copy_((torch.einsum("bhqk,bqhd->bkhd", ds, q) * scale).view(B, Sk, Hkv, g, d).sum(3))
    dv.copy_(torch.einsum("bhqk,bqhd->bkhd", p, do).view(B, Sk, Hkv, g, d).sum(3))


def _bwd_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    errs = []
    try:
        for layout in ("zigzag", "contiguous"):
            for causal in (True, False):
                g = torch.Generator().manual_seed(29 + world)
                B, S, Hq, Hkv, d = 2, 48, 4, 2, 8
                qf = torch.randn(B, S, Hq, d, generator=g, dtype=torch.float64)
                kf = torch.randn(B, S, Hkv, d, generator=g, dtype=torch.float64)
                vf = torch.randn(B, S, Hkv, d, generator=g, dtype=torch.float64)
                dof = torch.randn(B, S, Hq, d, generator=g, dtype=torch.float64)
                scale = 0.3
                qs, ks, vs, dos = (ring.split_sequence(t, world, rank, layout)
                                   for t in (qf, kf, vf, dof))
                fwd = ring.ring_forward(qs, ks, vs, causal, scale, layout=layout,
                                        attend=_oracle_attend, merge=_lse_merge)
                dq, dk, dv = ring.ring_backward(
                    qs, ks, vs, [o for o, _ in fwd], [lse for _, lse in fwd], dos, causal, scale,
                    layout=layout, backward=_pair_backward, accumulate=lambda a, x: a.add_(x),
                    finish=lambda a, out: out.copy_(a))
                rq, rk, rv = oracle.backward(qf, kf, vf, dof, scale, causal)
                c = S // ring.num_chunks(world, layout)
                for i, a in enumerate(ring.chunk_ids(world, rank, layout)):
                    rows = slice(a * c, (a + 1) * c)
                    for got, want in ((dq[i], rq), (dk[i], rk), (dv[i], rv)):
                        errs.append(float(np.abs(got.numpy() - want[:, rows]).max()))
        q.put((rank, max(errs)))
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_backward_on_gloo_ranks_equals_full_gradients(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_bwd_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _ in res] == list(range(world))
    for _, err in res:
        assert err <= 1e-12


def test_ring_backward_single_rank_equals_full_gradients():
    """world 1 (no process group): one pair per mask, no exchange."""
    import oracle
    g = torch.Generator().manual_seed(5)
    B, S, Hq, Hkv, d = 1, 32, 2, 1, 8
    qf, kf, vf, dof = (torch.randn(B, S, h, d, generator=g, dtype=torch.float64)
                       for h in (Hq, Hkv, Hkv, Hq))
    for causal in (True, False):
        qs, ks, vs, dos = (ring.split_sequence(t, 1, 0) for t in (qf, kf, vf, dof))
        fwd = ring.ring_forward(qs, ks, vs, causal, 0.5, attend=_oracle_attend,
                                merge=_lse_merge)
        dq, dk, dv = ring.ring_backward(
            qs, ks, vs, [o for o, _ in fwd], [lse for _, lse in fwd], dos, causal, 0.5,
            backward=_pair_backward, accumulate=lambda a, x: a.add_(x),
            finish=lambda a, out: out.copy_(a))
        rq, rk, rv = oracle.backward(qf, kf, vf, dof, 0.5, causal)
        c = S // 2
        for i, a in enumerate(ring.chunk_ids(1, 0)):
            rows = slice(a * c, (a + 1) * c)
            for got, want in ((dq[i], rq), (dk[i], rk), (dv[i], rv)):
                assert np.abs(got.numpy() - want[:, rows]).max() <= 1e-12
