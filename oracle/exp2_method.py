"""The exponential the attention kernels need, exactly and as the pages' method.

TEST INFRASTRUCTURE ONLY (see ``oracle/attention_fp64.py``). Shares no code and
no constants with the CUDA path.

* ``exp2_exact`` is the definition, 2**x in float64.
* ``exp2_range_reduced`` restates the software exponential of the pages
  ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
  Hardware Scaling", daily.dev Summary: a polynomial approximation evaluated on
  the FMA units after Cody-Waite range reduction). The input is already in
  base-2 units, so the reduction is exact: x = n + f with n = round(x) and
  f in [-1/2, 1/2], and 2**x = 2**n * 2**f. Only 2**f is approximated, by a
  polynomial of the given degree whose value at 0 is exactly 1; 2**n is applied
  exactly. The coefficients here are this module's own least-squares fit on
  Chebyshev nodes (a fit done at import, in float64), independent of whatever
  polynomial the CUDA path uses. The tests use it to show that the method, at a
  given degree, reaches a stated relative error; the CUDA exponential is then
  checked against ``exp2_exact`` directly.
"""
from __future__ import annotations

import numpy as np


def exp2_exact(x):
    return np.exp2(np.asarray(x, dtype=np.float64))


def fit_exp2_poly(degree: int, nodes: int = 512):
    """Least-squares fit of (2**f - 1)/f on [-1/2, 1/2] so that q(f) = 1 + f*r(f), q(0) = 1."""
    t = np.cos(np.pi * (np.arange(nodes) + 0.5) / nodes) * 0.5
    target = (np.exp2(t) - 1.0) / t
    # relative weighting: minimise the error of q relative to 2**f
    w = 1.0 / np.exp2(t)
    V = np.vander(t, degree, increasing=True)          # columns t^0 .. t^(degree-1)
    coef, *_ = np.linalg.lstsq(V * (w * t)[:, None], (target * t) * w, rcond=None)
    return np.concatenate([[1.0], coef])                 # q(f) = sum c_i f^i, c_0 = 1


def exp2_range_reduced(x, coeffs):
    """2**x as n = round(x), f = x - n, 2**n * q(f), in float64."""
    x = np.asarray(x, dtype=np.float64)
    n = np.rint(x)
    f = x - n
    q = np.zeros_like(f)
    for c in coeffs[::-1]:
        q = q * f + c
    return np.ldexp(q, n.astype(np.int64))
