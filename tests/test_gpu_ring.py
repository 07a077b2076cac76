"""Context-parallel ring with the library's kernels: two gloo ranks, both on
GPU 0, each running its own forwards and merges; K/V chunks move between
the ranks through host memory (gloo), so no kernel ever waits on another
rank. Each rank's merged O and LSE must match the fp64 oracle's attention over
the full sequence at that rank's rows (O max-abs 1e-2, LSE max-abs 1e-3, on
query heads {0, last}); the ring backward's dQ, dK, dV must match the oracle's
gradients over the full sequence at the rank's chunks (rel-L2 2e-2). The two
accumulation kernels it uses (fp32 += bf16, fp32 -> bf16) are checked bit for
bit against the same fp32 addition and round-to-nearest-even conversion."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    import exact_attention_smem_gb300 as fa
    import oracle
    from attn_inputs import random_inputs
    from exact_attention_smem_gb300 import ring
    res = []
    try:
        fa.load()
        x = random_inputs(B=1, Hq=8, Hkv=2, Sq=4096, Sk=4096, d=128, seed=300, device="cpu")
        for layout in ("zigzag", "contiguous"):
            for causal in (True, False):
                qs, ks, vs = (ring.split_sequence(t, world, rank, layout)
                              for t in (x.q, x.k, x.v))
                qs, ks, vs = ([t.cuda() for t in ts] for ts in (qs, ks, vs))
                out = ring.ring_forward(qs, ks, vs, causal, 128 ** -0.5, layout=layout)
                torch.cuda.synchronize()
                assert fa.fa_get_device_error(clear=True) == 0
                heads = [0, 7]
                ro, rl = oracle.forward(x.q, x.k, x.v, 128 ** -0.5, causal, heads=heads)
                c = 4096 // ring.num_chunks(world, layout)
                for (o, lse), a in zip(out, ring.chunk_ids(world, rank, layout)):
                    rows = slice(a * c, (a + 1) * c)
                    eo = np.abs(o.float().cpu().numpy()[:, :, heads] - ro[:, rows][:, :, heads]).max()
                    el = np.abs(lse.cpu().numpy()[:, heads] - rl[:, heads][:, :, rows]).max()
                    res.append((layout, causal, a, float(eo), float(el)))
        q.put((rank, res, None))
    except Exception as e:  # report instead of hanging the other rank's queue read
        q.put((rank, res, repr(e)))
    finally:
        dist.destroy_process_group()


def test_ring_two_ranks_one_gpu():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=120)
    for rank, res, err in out:
        assert err is None, (rank, err)
        assert len(res) == 6          # zigzag: 2 chunks x 2 masks, contiguous: 1 x 2
        for layout, causal, a, eo, el in res:
            assert eo <= 1e-2, (layout, causal, a, eo)
            assert el <= 1e-3, (layout, causal, a, el)
    assert all(p.exitcode == 0 for p in procs)


def _bwd_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    import exact_attention_smem_gb300 as fa
    import oracle
    from attn_inputs import random_inputs
    from exact_attention_smem_gb300 import ring
    from gpu_helpers import rel_l2
    res = []
    try:
        fa.load()
        S, d = 2048, 128
        x = random_inputs(B=1, Hq=4, Hkv=2, Sq=S, Sk=S, d=d, seed=301, device="cpu")
        for layout in ("zigzag", "contiguous"):
            for causal in (True, False):
                qs, ks, vs, dos = ([t.cuda() for t in ring.split_sequence(a, world, rank, layout)]
                                   for a in (x.q, x.k, x.v, x.do))
                fwd = ring.ring_forward(qs, ks, vs, causal, d ** -0.5, layout=layout)
                dq, dk, dv = ring.ring_backward(qs, ks, vs, [o for o, _ in fwd],
                                                [lse for _, lse in fwd], dos, causal, d ** -0.5,
                                                layout=layout)
                torch.cuda.synchronize()
                assert fa.fa_get_device_error(clear=True) == 0
                rq, rk, rv = oracle.backward(x.q, x.k, x.v, x.do, d ** -0.5, causal)
                c = S // ring.num_chunks(world, layout)
                for i, a in enumerate(ring.chunk_ids(world, rank, layout)):
                    rows = slice(a * c, (a + 1) * c)
                    errs = [rel_l2(got, want[:, rows])
                            for got, want in ((dq[i], rq), (dk[i], rk), (dv[i], rv))]
                    res.append((layout, causal, a, errs))
        q.put((rank, res, None))
    except Exception as e:  # report instead of hanging the other rank's queue read
        q.put((rank, res, repr(e)))
    finally:
        dist.destroy_process_group()


def test_ring_backward_two_ranks_one_gpu():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_bwd_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=120)
    for rank, res, err in out:
        assert err is None, (rank, err)
        assert len(res) == 6          # zigzag: 2 chunks x 2 masks, contiguous: 1 x 2
        for layout, causal, a, errs in res:
            assert max(errs) <= 2e-2, (layout, causal, a, errs)
            assert min(errs) > 0                          # the gradients were computed
    assert all(p.exitcode == 0 for p in procs)


@pytest.mark.parametrize("n", [8, 4096 * 8 + 8, 152 * 8 * 256 * 8 * 3 + 40])
def test_accumulate_and_conversion_bit_exact(n):
    """n spans one vector, a ragged count and several grid-stride passes."""
    import torch
    import exact_attention_smem_gb300 as fa
    g = torch.Generator(device="cpu").manual_seed(n)
    acc = (torch.randn(n, generator=g) * 3).cuda()
    x = (torch.randn(n, generator=g) * 0.01).to(torch.bfloat16).cuda()
    guard = torch.full((64,), 7.0, device="cuda")
    buf = torch.cat([acc, guard])
    want = acc + x.float()
    fa.fa_accumulate(buf, x, n)
    torch.cuda.synchronize()
    assert torch.equal(buf[:n], want)
    assert torch.equal(buf[n:], guard)                    # nothing written past n
    out = torch.full((n + 64,), 5.0, dtype=torch.bfloat16, device="cuda")
    fa.fa_to_bf16(out, buf, n)
    torch.cuda.synchronize()
    assert torch.equal(out[:n], want.to(torch.bfloat16))
    assert torch.equal(out[n:], torch.full((64,), 5.0, dtype=torch.bfloat16, device="cuda"))
    assert fa.fa_get_device_error(clear=True) == 0
