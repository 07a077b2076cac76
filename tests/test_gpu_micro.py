"""Microbenchmarks that size the exponential split and the tensor-core
denominator on the GPU at hand: MUFU ex2 vs the FMA-pipe polynomial
(exponentials per clock per SM) and tcgen05 bf16 MMA throughput (FLOP per clock
per SM). Results are printed and, when a ``gpurun_out/`` folder exists, saved
as JSON for the profile summaries."""
import json
import os

import pytest
import torch

import exact_attention_smem_gb300 as fa

pytestmark = pytest.mark.gpu


def _rate(kind, iters):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = torch.zeros(2 * sms, dtype=torch.float64, device="cuda")
    fa.fa_micro(kind, iters, out, sms)
    torch.cuda.synchronize()
    v = out.view(sms, 2).cpu()
    rates = v[:, 1] / v[:, 0]
    return float(rates.median()), sms


def test_microbenchmarks():
    fa.load()
    torch.cuda.set_device(0)
    fa.fa_get_device_error(clear=True)
    mufu, sms = _rate(0, 20000)
    poly, _ = _rate(1, 20000)
    mma, _ = _rate(2, 2000)
    assert fa.fa_get_device_error(clear=True) == 0
    res = {"sms": sms, "mufu_ex2_per_clk_per_sm": mufu, "poly_exp2_per_clk_per_sm": poly,
           "mma_bf16_flop_per_clk_per_sm": mma}
    print(json.dumps(res))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if os.path.isdir(os.path.join(root, "gpurun_out")):
        with open(os.path.join(root, "gpurun_out", "micro.json"), "w") as f:
            json.dump(res, f)
    assert 1 <= mufu <= 256 and 1 <= poly <= 256
    assert 1000 <= mma <= 65536
