"""Microbenchmarks that size the exponential split and the tensor-core
denominator on the GPU at hand: MUFU ex2 vs the FMA-pipe polynomial
(exponentials per clock per SM) and tcgen05 bf16 MMA throughput (FLOP per clock
per SM). Results are printed and, when the environment variable FA_MICRO_OUT
names a directory, saved there as micro.json for the profile summaries."""
import json
import os

import pytest
import torch

import exact_attention_smem_gb300 as fa
import fa_testing_lib as ft

pytestmark = pytest.mark.gpu


def _rate(kind, iters):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = torch.zeros(2 * sms, dtype=torch.float64, device="cuda")
    ft.fa_micro(kind, iters, out, sms)
    torch.cuda.synchronize()
    v = out.view(sms, 2).cpu()
    rates = v[:, 1] / v[:, 0]
    return float(rates.median()), sms


def test_microbenchmarks():
    fa.load()
    torch.cuda.set_device(0)
    ft.fa_test_get_device_error(clear=True)
    mufu, sms = _rate(0, 20000)
    poly, _ = _rate(1, 20000)
    mma, _ = _rate(2, 2000)
    shapes = {name: _rate(kind, 2000)[0] for kind, name in
              ((3, "ss_n128"), (4, "ss_n64"), (5, "ts_n128"), (6, "ts_n64"),
               (7, "elect_ss_n256"), (8, "elect_ss_n128"), (9, "elect_ss_n64"),
               (10, "elect_ts_n128"), (11, "elect_ts_n64"))}
    issue = {f"mods{m}": _rate(12 + m, 2000)[0] for m in (0, 1, 2, 4, 8, 15)}
    issue.update({name: _rate(kind, 2000)[0] for kind, name in
                  ((28, "lane0_inloop_desc"), (29, "elect_inloop_desc"), (30, "lane0_hoisted_desc"),
                   (31, "lane0_runtime_acc"), (32, "lane0_fence"), (33, "lane0_commit"),
                   (34, "lane0_mbar_wait"), (35, "lane0_bare_try_wait"),
                   (36, "lane0_test_wait"), (37, "elect_named_barrier"),
                   (38, "lane0_smem_flag"), (39, "lane0_global_read"))})
    lat = {}
    for op, oname in ((0, "tmem_ld"), (1, "smem_ld"), (2, "mbar_test")):
        for same in (0, 1):
            for busy in (0, 1):
                r, _ = _rate(40 + op * 4 + same * 2 + busy, 2000)
                lat[f"{oname}_{'same' if same else 'other'}_sub_{'mma' if busy else 'idle'}"] = 1.0 / r
    assert ft.fa_test_get_device_error(clear=True) == 0
    res = {"probe_latency_clk": lat, "issue_ss_n128_by_extras": issue,"sms": sms, "mufu_ex2_per_clk_per_sm": mufu, "poly_exp2_per_clk_per_sm": poly,
           "mma_bf16_flop_per_clk_per_sm": mma,
           "mma_flop_per_clk_per_sm_by_shape": dict(ss_n256=mma, **shapes)}
    print(json.dumps(res))
    out_dir = os.environ.get("FA_MICRO_OUT")
    if out_dir and os.path.isdir(out_dir):
        with open(os.path.join(out_dir, "micro.json"), "w") as f:
            json.dump(res, f)
    assert 1 <= mufu <= 256 and 1 <= poly <= 256
    assert 1000 <= mma <= 65536
