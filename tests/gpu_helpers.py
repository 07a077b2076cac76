"""Shared helpers for the GPU parity tests (comparison metrics, guarded buffers)."""
import math

import numpy as np
import torch

O_TOL = 1e-2      # O max-abs error vs the fp64 oracle
LSE_TOL = 1e-3    # LSE max-abs error
GRAD_TOL = 2e-2   # dQ/dK/dV relative L2 error

SENTINEL = -12345.0


def guarded(shape, dtype, device, margin=4096):
    """A tensor view inside a larger buffer whose margins hold a sentinel value."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * margin,), SENTINEL, dtype=dtype, device=device)
    view = buf[margin:margin + n].view(*shape)
    return buf, view


def margins_intact(buf, margin=4096):
    head = buf[:margin].float()
    tail = buf[-margin:].float()
    s = torch.tensor(SENTINEL, dtype=buf.dtype).float().item()
    return bool((head == s).all()) and bool((tail == s).all())


def max_abs(got, ref):
    """Largest |got - ref| over the entries the oracle computed (ref not NaN).

    Matching infinities (fully masked rows: LSE = +inf) count as zero error; a
    NaN or a mismatched infinity in `got` counts as infinite error.
    """
    g = got.detach().float().cpu().numpy().astype(np.float64)
    sel = ~np.isnan(ref)
    g, r = g[sel], ref[sel]
    same_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore"):                  # inf - inf where both are +inf
        d = np.where(same_inf, 0.0, np.abs(g - r))
    d = np.where(np.isnan(d), np.inf, d)
    return float(d.max()) if d.size else 0.0


def rel_l2(got, ref, floor_rms=1e-3):
    """||got - ref||_2 / ||ref||_2 over the entries the oracle computed.

    The denominator has a floor of `floor_rms` * sqrt(n): where the exact
    gradient is (near) zero — e.g. a single visible key makes dS, hence dQ and
    dK, exactly 0 — the check becomes an absolute RMS bound instead of a ratio
    of rounding noise to zero.
    """
    g = got.detach().float().cpu().numpy().astype(np.float64)
    sel = ~np.isnan(ref)
    g, r = g[sel], ref[sel]
    denom = max(float(np.linalg.norm(r)), floor_rms * math.sqrt(max(r.size, 1)))
    return float(np.linalg.norm(g - r) / denom)
