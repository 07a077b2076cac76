"""Context parallelism: attention over a sequence split across ranks (a ring).

The keys and values of a long sequence are split into chunks held by
different ranks; every rank keeps its query chunks and passes its K/V chunks
around a ring of ranks, so that after N steps each rank has seen every K/V
chunk once. For each (query chunk, received key chunk) pair that has visible
keys the rank runs one forward (``fa_fwd``), keeping O and the row
log-sum-exp; at the end ``fa_merge`` combines the parts of each query chunk
into the attention over all keys. This is exact: merging by the log-sum-exp
is the online-softmax rescale applied across parts ("FlashAttention-4
Conquers Asymmetric GPU Hardware Scaling", episode description: tiling with an
online softmax; its source list names Ring Attention, blockwise attention
across devices).

Chunk layout. The sequence (length S, every batch entry and head alike) is cut
into 2N equal chunks of c = S / (2N) rows; rank r holds global chunks r and
2N - 1 - r ("zigzag"), so that under a causal mask every rank has the same
amount of work. ``contiguous`` layout (one chunk per rank, rank r holds chunk
r) is also available. A query chunk a and a key chunk b give:
  * non-causal: every key visible (an Sq = Sk = c forward, no mask);
  * causal, b < a: every key visible (no mask);
  * causal, b == a: the diagonal block (a causal forward, Sq = Sk = c);
  * causal, b > a: no visible key (skipped).

Exchange. Each step sends the rank's current K/V chunks to rank r + 1 and
receives rank r - 1's with non-blocking point-to-point operations posted
before the step's forwards, so the transfer overlaps the compute. With the
NCCL backend device tensors move directly; with gloo (CPU ranks, or a test)
they are staged through host memory. No TMA or kernel ever reads a peer's
memory.

The forward and merge are the library's kernels (``attend`` / ``merge``
default to them); they are parameters so that the ring's schedule can be
checked on CPU ranks against a reference.
"""
from __future__ import annotations

import math


def chunk_ids(world: int, rank: int, layout: str = "zigzag") -> list[int]:
    """Global chunk indices held by `rank` (in the order of its local chunks)."""
    if layout == "zigzag":
        return [rank, 2 * world - 1 - rank]
    if layout == "contiguous":
        return [rank]
    raise ValueError(f"unknown layout {layout!r}")


def num_chunks(world: int, layout: str = "zigzag") -> int:
    return 2 * world if layout == "zigzag" else world


def split_sequence(x, world: int, rank: int, layout: str = "zigzag", dim: int = 1):
    """The chunks of a full [B, S, H, d] tensor that `rank` holds (contiguous copies)."""
    n = num_chunks(world, layout)
    S = x.shape[dim]
    if S % n:
        raise ValueError(f"sequence length {S} is not a multiple of {n} chunks")
    c = S // n
    return [x.narrow(dim, i * c, c).contiguous() for i in chunk_ids(world, rank, layout)]


def pair_mask(q_chunk: int, k_chunk: int, causal: bool):
    """'full', 'causal' (the diagonal block) or None (no visible key)."""
    if not causal or k_chunk < q_chunk:
        return "full"
    if k_chunk == q_chunk:
        return "causal"
    return None


def _fa_attend(q, k, v, causal, scale, out, lse):
    from . import forward
    forward(q, k, v, causal=causal, scale=scale, out=out, lse=lse)


def _fa_merge(o_parts, lse_parts):
    """Merge P parts (o_parts [P, B, S, H, d] bf16, lse_parts [P, B, H, S] fp32)."""
    import torch
    from ._lib import fa_merge
    P, B, S, H, d = o_parts.shape
    o = torch.empty(o_parts.shape[1:], dtype=o_parts.dtype, device=o_parts.device)
    lse = torch.empty(lse_parts.shape[1:], dtype=lse_parts.dtype, device=lse_parts.device)
    fa_merge(o_parts, lse_parts, P, B, H, S, d, 0, o, lse)
    return o, lse


def ring_schedule(world: int, rank: int, causal: bool, layout: str = "zigzag"):
    """The forwards `rank` runs, step by step: a list over steps of
    (source rank, [(local query chunk, local key chunk of the source, mask), ...])."""
    mine = chunk_ids(world, rank, layout)
    steps = []
    for step in range(world):
        src = (rank - step) % world
        pairs = []
        for qi, a in enumerate(mine):
            for ki, b in enumerate(chunk_ids(world, src, layout)):
                m = pair_mask(a, b, causal)
                if m is not None:
                    pairs.append((qi, ki, m))
        steps.append((src, pairs))
    return steps


def ring_forward(q_chunks, k_chunks, v_chunks, causal: bool, scale: float | None = None,
                 group=None, layout: str = "zigzag", attend=None, merge=None):
    """Attention of this rank's query chunks over the whole sequence's keys.

    q_chunks, k_chunks, v_chunks: this rank's chunks (see ``split_sequence``),
    each [B, c, H, d] (k/v with Hkv heads). Every rank of `group` calls this
    with the same layout and chunk length. Returns a list with (O, LSE) per
    query chunk: O [B, c, Hq, d], LSE [B, Hq, c] (natural log, fa_fwd's
    convention). The parts of each query chunk are written straight into the
    buffers the merge reads.
    """
    import torch
    import torch.distributed as dist

    attend = attend or _fa_attend
    merge = merge or _fa_merge
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if scale is None:
        scale = 1.0 / math.sqrt(q_chunks[0].shape[-1])
    nloc = len(chunk_ids(world, rank, layout))
    if len(q_chunks) != nloc or len(k_chunks) != nloc or len(v_chunks) != nloc:
        raise ValueError(f"rank {rank} holds {nloc} chunks in the {layout} layout")
    schedule = ring_schedule(world, rank, causal, layout)
    staged = (world > 1 and dist.get_backend(group) == "gloo" and q_chunks[0].is_cuda)
    device = q_chunks[0].device
    # one O / LSE slot per (query chunk, visible key chunk)
    nparts = [0] * nloc
    for _, pairs in schedule:
        for qi, _, _ in pairs:
            nparts[qi] += 1
    # LSE in fp32 for bf16/fp16 inputs (fa_fwd's output), else in the inputs' type
    lse_dtype = torch.float32 if q_chunks[0].dtype in (torch.bfloat16, torch.float16) \
        else q_chunks[0].dtype
    o_parts, lse_parts = [], []
    for qi, q in enumerate(q_chunks):
        B, c, H, d = q.shape
        if (B * H * c) % 4:
            raise ValueError("B * Hq * chunk length must be a multiple of 4 (16-byte aligned "
                             "LSE parts)")
        o_parts.append(torch.empty((nparts[qi], B, c, H, v_chunks[0].shape[-1]), dtype=q.dtype,
                                   device=device))
        lse_parts.append(torch.empty((nparts[qi], B, H, c), dtype=lse_dtype, device=device))
    filled = [0] * nloc

    cur = [t.cpu() if staged else t for t in list(k_chunks) + list(v_chunks)]
    nxt_rank, prv_rank = (rank + 1) % world, (rank - 1) % world
    for step, (src, pairs) in enumerate(schedule):
        reqs, incoming = [], None
        if step + 1 < world:
            incoming = [torch.empty_like(t) for t in cur]
            for t in cur:
                reqs.append(dist.isend(t, dst=_global(nxt_rank, group), group=group))
            for t in incoming:
                reqs.append(dist.irecv(t, src=_global(prv_rank, group), group=group))
        kv = [t.to(device, non_blocking=True) for t in cur] if staged else cur
        ks, vs = kv[:nloc], kv[nloc:]
        for qi, ki, m in pairs:
            slot = filled[qi]
            attend(q_chunks[qi], ks[ki], vs[ki], m == "causal", scale, o_parts[qi][slot],
                   lse_parts[qi][slot])
            filled[qi] += 1
        for r in reqs:
            r.wait()
        if incoming is not None:
            cur = incoming
    return [merge(o_parts[qi], lse_parts[qi]) for qi in range(nloc)]


def _global(rank_in_group, group):
    import torch.distributed as dist
    if group is None:
        return rank_in_group
    return dist.get_global_rank(group, rank_in_group)
