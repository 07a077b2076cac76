"""fp64 CPU restatement of the tiled online softmax with conditional rescaling.

TEST INFRASTRUCTURE ONLY (see ``oracle/attention_fp64.py``). Shares no code with
the CUDA path.

Steps, in the order the pages give them:

* Tiling plus online softmax ("FlashAttention-4 Conquers Asymmetric GPU Hardware
  Scaling", episode description, lineage paragraph): walk the keys one block at
  a time, keeping per row a running maximum and a running sum, so the score
  matrix is never materialised.
* Conditional online-softmax rescaling ("FlashAttention-4: Algorithm and Kernel
  Pipelining Co-Design for Asymmetric Hardware Scaling", daily.dev Summary;
  same technique in the abstract, item (2)): the accumulator is rescaled only
  when a row's running maximum has grown past a threshold ``tau``; otherwise the
  stale reference maximum is kept. In exact arithmetic the result does not
  depend on ``tau`` (the reading taken here: the test is ``m_new > m_ref + tau``
  per row, in natural-log units).

This is a check of the *algorithm* against the plain definition in
``attention_fp64.attend_head``: both are fp64, so they agree to rounding.
"""
from __future__ import annotations

import numpy as np


def online_attend_head(q, k, v, scale: float, causal: bool, block_n: int = 128,
                       tau: float = 0.0, return_stats: bool = False):
    """Tiled forward for one (sequence, head): returns (o, lse) [, rescale count]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, nk = q.shape[0], k.shape[0]
    m_ref = np.full(nq, -np.inf)      # reference maximum used for the exponentials
    l = np.zeros(nq)                  # running sum of exp(s - m_ref)
    acc = np.zeros((nq, v.shape[1]))  # running sum of exp(s - m_ref) * v
    rescales = 0
    rows = np.arange(nq)[:, None]
    for j0 in range(0, nk, block_n):
        j1 = min(nk, j0 + block_n)
        s = scale * (q @ k[j0:j1].T)
        if causal:
            cols = np.arange(j0, j1)[None, :]
            s = np.where(cols <= rows + (nk - nq), s, -np.inf)
        m_blk = s.max(axis=1)
        grow = m_blk > m_ref + tau    # -inf + tau = -inf: the first visible block always "grows"
        m_new = np.where(grow, m_blk, m_ref)
        alpha = np.where(np.isfinite(m_ref) & grow, np.exp(m_ref - m_new), 1.0)
        alpha = np.where(np.isfinite(m_ref), alpha, 0.0)
        rescales += int(np.count_nonzero(grow & np.isfinite(m_ref)))
        acc *= alpha[:, None]
        l *= alpha
        m_ref = m_new
        m_sub = np.where(np.isfinite(m_ref), m_ref, 0.0)
        p = np.exp(s - m_sub[:, None])
        l += p.sum(axis=1)
        acc += p @ v[j0:j1]
    has = l > 0
    o = np.where(has[:, None], acc / np.where(has, l, 1.0)[:, None], 0.0)
    lse = np.where(has, m_ref + np.log(np.where(has, l, 1.0)), np.inf)
    if return_stats:
        return o, lse, rescales
    return o, lse
