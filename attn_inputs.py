"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark. It draws random numbers and lays them out; it holds none of the
attention arithmetic.

Recipe (one ``torch.Generator(device="cpu").manual_seed(seed)`` per workload):

* varlen only: first draw the sequence lengths, ``L_i = round(exp(U[ln lo, ln hi]))``
  (``torch.rand`` in float64);
* then Q, K, V, dO in that order with ``torch.randn(..., dtype=float32)``;
* GQA workload only: then one factor ``f_g ~ U[0.5, 2]`` per KV head; K rows of
  head g are multiplied by ``f_g`` in float32 (``scale_v=True`` also scales V);
* finally every tensor is rounded to bfloat16 (round-to-nearest-even).

Dense tensors are ``[B, S, H, d]``; packed variable-length tensors are
``[T, H, d]`` with int32 ``cu_seqlens`` of length ``nseq + 1``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    d: int
    causal: bool
    seed: int
    backward: bool = True
    varlen_nseq: int = 0          # >0: packed variable-length batch
    varlen_lo: int = 128
    varlen_hi: int = 16384
    kv_head_factors: bool = False  # per-KV-head factor U[0.5, 2] on K rows
    scale_v: bool = False          # also apply the factor to V rows
    scale: float = field(default=0.0)

    def __post_init__(self):
        if self.scale == 0.0:
            self.scale = 1.0 / math.sqrt(self.d)


# The five workloads: shapes, masks and seeds.
WORKLOADS = {
    "fwd_small_d64": Workload("fwd_small_d64", B=1, Hq=2, Hkv=2, Sq=256, Sk=256, d=64,
                              causal=False, seed=0, backward=False),
    "mha_s2048": Workload("mha_s2048", B=4, Hq=16, Hkv=16, Sq=2048, Sk=2048, d=128,
                          causal=False, seed=1),
    "mha_s2048_causal": Workload("mha_s2048_causal", B=4, Hq=16, Hkv=16, Sq=2048, Sk=2048,
                                 d=128, causal=True, seed=1),
    "long_s32768_causal": Workload("long_s32768_causal", B=1, Hq=32, Hkv=32, Sq=32768,
                                   Sk=32768, d=128, causal=True, seed=2),
    "gqa_s8192_causal": Workload("gqa_s8192_causal", B=8, Hq=64, Hkv=8, Sq=8192, Sk=8192,
                                 d=128, causal=True, seed=3, kv_head_factors=True),
    "varlen16_causal": Workload("varlen16_causal", B=16, Hq=32, Hkv=32, Sq=16384, Sk=16384,
                                d=128, causal=True, seed=4, varlen_nseq=16),
}


def varlen_lengths(gen: torch.Generator, nseq: int, lo: int, hi: int) -> list[int]:
    """Log-uniform lengths on [lo, hi], drawn first from the workload's generator."""
    u = torch.rand(nseq, generator=gen, dtype=torch.float64)
    lengths = torch.round(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return [int(x) for x in lengths.tolist()]


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    cu_seqlens: torch.Tensor | None
    lengths: list[int] | None
    kv_factors: list[float] | None
    cu_seqlens_k: torch.Tensor | None = None   # key boundaries, when they differ from cu_seqlens


def make_inputs(w: Workload, device: str | torch.device = "cpu") -> Inputs:
    """Draw the workload's bf16 tensors (on the CPU, then moved to ``device``)."""
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    lengths = None
    cu = None
    if w.varlen_nseq:
        lengths = varlen_lengths(gen, w.varlen_nseq, w.varlen_lo, w.varlen_hi)
        T = sum(lengths)
        qs, ks = (T, w.Hq, w.d), (T, w.Hkv, w.d)
        cu = torch.tensor([0] + list(_cumsum(lengths)), dtype=torch.int32)
    else:
        qs, ks = (w.B, w.Sq, w.Hq, w.d), (w.B, w.Sk, w.Hkv, w.d)
    q = torch.randn(qs, generator=gen, dtype=torch.float32)
    k = torch.randn(ks, generator=gen, dtype=torch.float32)
    v = torch.randn(ks, generator=gen, dtype=torch.float32)
    do = torch.randn(qs, generator=gen, dtype=torch.float32)
    factors = None
    if w.kv_head_factors:
        f = torch.rand(w.Hkv, generator=gen, dtype=torch.float32) * 1.5 + 0.5
        factors = [float(x) for x in f.tolist()]
        k = k * f.view(*([1] * (k.dim() - 2)), w.Hkv, 1)
        if w.scale_v:
            v = v * f.view(*([1] * (v.dim() - 2)), w.Hkv, 1)
    out = [t.to(torch.bfloat16).to(device) for t in (q, k, v, do)]
    if cu is not None:
        cu = cu.to(device)
    return Inputs(*out, cu_seqlens=cu, lengths=lengths, kv_factors=factors)


def random_inputs(B, Hq, Hkv, Sq, Sk, d, seed, lengths=None, device="cpu", std=1.0,
                  lengths_k=None):
    """Small ad-hoc cases for tests (same draw order as the workloads).

    lengths_k (packed only): per-sequence key counts, giving k/v their own
    rows [Tk, Hkv, d] and boundary list (cu_seqlens_k)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    cu_k = None
    if lengths is not None:
        T = sum(lengths)
        Tk = T if lengths_k is None else sum(lengths_k)
        qs, ks = (T, Hq, d), (Tk, Hkv, d)
        cu = torch.tensor([0] + list(_cumsum(lengths)), dtype=torch.int32)
        if lengths_k is not None:
            cu_k = torch.tensor([0] + list(_cumsum(lengths_k)), dtype=torch.int32)
    else:
        qs, ks = (B, Sq, Hq, d), (B, Sk, Hkv, d)
        cu = None
    q = torch.randn(qs, generator=gen, dtype=torch.float32) * std
    k = torch.randn(ks, generator=gen, dtype=torch.float32) * std
    v = torch.randn(ks, generator=gen, dtype=torch.float32)
    do = torch.randn(qs, generator=gen, dtype=torch.float32)
    out = [t.to(torch.bfloat16).to(device) for t in (q, k, v, do)]
    if cu is not None:
        cu = cu.to(device)
    if cu_k is not None:
        cu_k = cu_k.to(device)
    return Inputs(*out, cu_seqlens=cu, lengths=lengths, kv_factors=None, cu_seqlens_k=cu_k)


def _cumsum(xs):
    s = 0
    for x in xs:
        s += x
        yield s


def flops_forward(w: Workload, lengths: list[int] | None = None) -> float:
    """Forward FLOPs: 4*B*Hq*Sq*Sk*d, halved for causal; varlen sums per sequence."""
    if lengths is not None:
        tot = sum(4.0 * w.Hq * L * L * w.d for L in lengths)
    else:
        tot = 4.0 * w.B * w.Hq * w.Sq * w.Sk * w.d
    return tot / 2 if w.causal else tot
