"""fp64 CPU oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this module. The CUDA path
never calls it, and it shares no code with the CUDA path.

What it computes, and where that is defined
-------------------------------------------
The method is *exact* attention: the tiled, online-softmax kernels must give the
same result as the plain definition ("FlashAttention-4 Conquers Asymmetric GPU
Hardware Scaling", episode description, lineage paragraph: tiling and online
softmax avoid materialising the N x N score matrix; the result is unchanged).
So this oracle is that plain definition, materialising the scores in float64:

forward, per sequence and query head h (KV head g = h // (Hq // Hkv)):
    S    = scale * Q_h K_g^T                         (Sq x Sk)
    S_ij = -inf  where causal and j > i + (Sk - Sq)  (bottom-right alignment)
    m_i  = max_j S_ij ;  p_ij = exp(S_ij - m_i) ;  l_i = sum_j p_ij
    O_h  = (p V_g) / l ;  LSE_i = m_i + ln(l_i)      (natural log, scaled scores)
    rows with no visible key: O = 0, LSE = +inf

backward (the exact gradient of the forward above, given dO):
    P  = exp(S - LSE) ; dP = dO_h V_g^T ; D_i = sum_j P_ij dP_ij
    dS = P * (dP - D)
    dQ_h = scale * dS K_g ; dK_g += scale * dS^T Q_h ; dV_g += P^T dO_h

The query rows are processed in chunks (``row_chunk``) only to bound memory;
each row still gets the full two-pass softmax over all of its keys.

Layouts: dense ``[B, S, H, d]``; packed variable-length ``[T, H, d]`` with
``cu_seqlens`` (one boundary list for queries and keys, or, with
``cu_seqlens_k``, separate lists: sequence i's queries are rows
[cu_seqlens[i], cu_seqlens[i+1]) of q and its keys rows
[cu_seqlens_k[i], cu_seqlens_k[i+1]) of k and v, causal bottom-right aligned
per sequence). LSE is ``[B, Hq, Sq]`` dense or ``[Hq, Tq]`` packed.
"""
from __future__ import annotations

import numpy as np


def _as64(x):
    """Accept numpy arrays or torch tensors (any float dtype); return float64 numpy."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()     # exact for bf16, fp16, fp32 and fp64
    return np.asarray(x, dtype=np.float64)


def _visible(nq: int, nk: int, causal: bool, row0: int = 0, rows: int | None = None):
    """Boolean visibility mask for query rows [row0, row0+rows) against all keys."""
    rows = nq - row0 if rows is None else rows
    if not causal:
        return np.ones((rows, nk), dtype=bool)
    i = np.arange(row0, row0 + rows)[:, None]
    j = np.arange(nk)[None, :]
    return j <= i + (nk - nq)


def attend_head(q, k, v, scale: float, causal: bool, row_chunk: int = 1024,
                return_max: bool = False):
    """Forward for one (sequence, query head): q [Sq, d], k/v [Sk, d] -> (o [Sq, d], lse [Sq]).

    With ``return_max`` also the row maxima m [Sq] of the scaled, masked scores
    (the m_i of the definition above; -inf for a row with no visible key)."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    nq, nk = q.shape[0], k.shape[0]
    o = np.zeros((nq, v.shape[1]))
    lse = np.full(nq, np.inf)
    mx = np.full(nq, -np.inf)
    for r0 in range(0, nq, row_chunk):
        r1 = min(nq, r0 + row_chunk)
        s = scale * (q[r0:r1] @ k.T)
        vis = _visible(nq, nk, causal, r0, r1 - r0)
        s = np.where(vis, s, -np.inf)
        m = s.max(axis=1, initial=-np.inf)        # -inf also for a sequence with no keys
        has = np.isfinite(m)
        m_safe = np.where(has, m, 0.0)
        p = np.exp(s - m_safe[:, None])
        l = p.sum(axis=1)
        o[r0:r1] = np.where(has[:, None], (p @ v) / np.where(has, l, 1.0)[:, None], 0.0)
        lse[r0:r1] = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), np.inf)
        mx[r0:r1] = m
    return (o, lse, mx) if return_max else (o, lse)


def attend_head_backward(q, k, v, do, scale: float, causal: bool, row_chunk: int = 1024):
    """Backward for one (sequence, query head).

    Returns (dq [Sq, d], dk [Sk, d], dv [Sk, d]) — dk/dv are this head's
    contribution (the caller sums them over the heads of a KV group).
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    _, lse = attend_head(q, k, v, scale, causal, row_chunk)
    nq, nk = q.shape[0], k.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, nq, row_chunk):
        r1 = min(nq, r0 + row_chunk)
        s = scale * (q[r0:r1] @ k.T)
        vis = _visible(nq, nk, causal, r0, r1 - r0)
        s = np.where(vis, s, -np.inf)
        p = np.exp(s - lse[r0:r1, None])          # exp(-inf) = 0, also for LSE = +inf rows
        dp = do[r0:r1] @ v.T
        dsum = (p * dp).sum(axis=1)
        ds = p * (dp - dsum[:, None])
        dq[r0:r1] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r0:r1])
        dv += p.T @ do[r0:r1]
    return dq, dk, dv


def _bounds(cu):
    return [int(x) for x in (cu.tolist() if hasattr(cu, "tolist") else cu)]


def _segments(q, cu_seqlens, cu_seqlens_k=None):
    """Yield (seq index, q row slice, k row slice) for dense or packed layouts."""
    if cu_seqlens is None:
        for b in range(q.shape[0]):
            yield b, (b, slice(None)), (b, slice(None))
    else:
        cu = _bounds(cu_seqlens)
        ck = cu if cu_seqlens_k is None else _bounds(cu_seqlens_k)
        for i in range(len(cu) - 1):
            yield i, (slice(cu[i], cu[i + 1]),), (slice(ck[i], ck[i + 1]),)


def forward(q, k, v, scale: float, causal: bool, cu_seqlens=None, heads=None, seqs=None,
            row_chunk: int = 1024, cu_seqlens_k=None):
    """Forward over a whole batch (or a subset of query heads / sequences).

    Returns (o, lse) as float64 arrays in the caller's layout; entries of heads or
    sequences not in the subset are NaN.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    hq, hkv = q.shape[-2], k.shape[-2]
    group = hq // hkv
    o = np.full(q.shape[:-1] + (v.shape[-1],), np.nan)
    if cu_seqlens is None:
        lse = np.full((q.shape[0], hq, q.shape[1]), np.nan)
    else:
        lse = np.full((hq, q.shape[0]), np.nan)
    heads = range(hq) if heads is None else heads
    for si, qi, ki in _segments(q, cu_seqlens, cu_seqlens_k):
        if seqs is not None and si not in seqs:
            continue
        for h in heads:
            g = h // group
            oh, lh = attend_head(q[qi][..., h, :], k[ki][..., g, :], v[ki][..., g, :], scale,
                                 causal, row_chunk)
            o[qi + (h,)] = oh
            if cu_seqlens is None:
                lse[si, h] = lh
            else:
                lse[h, qi[0]] = lh
    return o, lse


def backward(q, k, v, do, scale: float, causal: bool, cu_seqlens=None, kv_heads=None,
             seqs=None, row_chunk: int = 1024, cu_seqlens_k=None):
    """Backward over a whole batch (or a subset of KV heads / sequences).

    For each selected KV head g, all query heads of its group contribute to dK_g
    and dV_g. Returns (dq, dk, dv) in the caller's layout; unselected entries NaN.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    hq, hkv = q.shape[-2], k.shape[-2]
    group = hq // hkv
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    kv_heads = range(hkv) if kv_heads is None else kv_heads
    for si, qi, ki in _segments(q, cu_seqlens, cu_seqlens_k):
        if seqs is not None and si not in seqs:
            continue
        for g in kv_heads:
            acc_k = np.zeros(k[ki][..., g, :].shape)
            acc_v = np.zeros(v[ki][..., g, :].shape)
            for h in range(g * group, (g + 1) * group):
                dqh, dkh, dvh = attend_head_backward(q[qi][..., h, :], k[ki][..., g, :],
                                                     v[ki][..., g, :], do[qi][..., h, :],
                                                     scale, causal, row_chunk)
                dq[qi + (h,)] = dqh
                acc_k += dkh
                acc_v += dvh
            dk[ki + (g,)] = acc_k
            dv[ki + (g,)] = acc_v
    return dq, dk, dv
