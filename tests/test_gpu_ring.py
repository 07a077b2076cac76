"""Context-parallel ring with the library's kernels: two gloo ranks, both on
GPU 0, each running its own forwards and merges; K/V chunks move between
the ranks through host memory (gloo), so no kernel ever waits on another
rank. Each rank's merged O and LSE must match the fp64 oracle's attention over
the full sequence at that rank's rows (O max-abs 1e-2, LSE max-abs 1e-3, on
query heads {0, last})."""
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
