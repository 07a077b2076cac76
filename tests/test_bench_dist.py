"""The benchmark's multi-rank aggregation (max of per-rank times, whole-job
throughput) on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 100.0 + 50.0 * rank
    ms = bench.max_over_ranks(ms_local)
    q.put((rank, ms, bench.job_tflops(1e12, 10, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tf in res:
        assert ms == 150.0                      # the slowest rank's time
        assert tf == pytest.approx(1e12 * 10 * 2 / 0.150 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(2e12, 5, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_json_contract():
    """`bench.py --impl reference` (the fp64 oracle on the host cores, a
    bounded sample per step) prints one JSON line with the bench contract's
    keys, its own e2e with no host-device bytes and a cpu_baseline entry."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--workload", "mha_s2048_causal"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in out, key
    assert out["impl"] == "reference" and out["value"] > 0 and out["unit"] == "TFLOP/s"
    assert out["higher_is_better"] is True and out["dtype"] == "f64"
    assert out["config"]["workload"] == "mha_s2048_causal"
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["value"] == out["value"]
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["d2h_bytes_per_step"] == 0
