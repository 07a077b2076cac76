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

Backward (``ring_backward``). With the merged O and LSE of its query rows, a
(query chunk a, key chunk b) pair's share of the gradients is exactly what
``fa_bwd`` computes for that pair alone: P = exp(S - LSE) uses the LSE over
all keys and D = rowsum(dO * O) the merged O, so the pair's dQ_a, dK_b and dV_b
are the terms of the full sums that involve the pair's keys ("FlashAttention-4:
Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling",
abstract item 3: the backward recomputes P from the saved LSE and accumulates
dQ over key blocks). The K/V chunks go around the ring as in the forward, and
their dK/dV sums (fp32 for bf16 inputs) travel one step behind them: a rank
adds its pairs' dK/dV into the sums it received, then passes them on, so the
transfer of a sum overlaps the next step's backwards; after the last step
each sum has visited every rank and arrives at the rank that owns the chunk.
dQ sums stay local. The sums are kept in fp32 by two small library kernels
(``fa_accumulate``: fp32 += bf16, ``fa_to_bf16``).

The forward, backward, merge and accumulation are the library's kernels
(``attend`` / ``merge`` / ``backward`` / ``accumulate`` / ``finish`` default to
them); they are parameters so that the ring's schedule and exchange can be
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


def _fa_backward():
    """Per-pair backward into the caller's buffers, with one reused workspace."""
    import torch
    from ._lib import fa_bwd, fa_bwd_workspace_bytes
    ws = [None]

    def backward(q, k, v, o, lse, do, causal, scale, dq, dk, dv):
        B, Sq, Hq, d = q.shape
        Sk, Hkv = k.shape[1], k.shape[2]
        nbytes = fa_bwd_workspace_bytes(B, Hq, Sq, d, 0)
        if ws[0] is None or ws[0].numel() < nbytes:
            ws[0] = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        fa_bwd(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale, None,
               ws[0], nbytes, None)
    return backward


def _fa_accumulate(acc, x):
    from ._lib import fa_accumulate
    fa_accumulate(acc, x)


def _fa_finish(acc, out):
    from ._lib import fa_to_bf16
    fa_to_bf16(out, acc)


_TAG_KV, _TAG_ACC = 1, 2


def _exchange(send, recv, nxt, prv, group, tag):
    """Post sends of `send` to rank `nxt` and receives into `recv` from rank
    `prv` as one batch (one NCCL group: no ordering deadlock when nxt == prv)."""
    import torch.distributed as dist
    ops = [dist.P2POp(dist.isend, t, _global(nxt, group), group, tag) for t in send]
    ops += [dist.P2POp(dist.irecv, t, _global(prv, group), group, tag) for t in recv]
    return dist.batch_isend_irecv(ops)


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
            reqs = _exchange(cur, incoming, nxt_rank, prv_rank, group, _TAG_KV)
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


def ring_backward(q_chunks, k_chunks, v_chunks, o_chunks, lse_chunks, do_chunks, causal: bool,
                  scale: float | None = None, group=None, layout: str = "zigzag", backward=None,
                  accumulate=None, finish=None):
    """dQ, dK, dV of this rank's chunks for attention over the whole sequence.

    q/k/v_chunks as for ``ring_forward``; o_chunks and lse_chunks are the
    merged outputs ``ring_forward`` returned for this rank's query chunks
    ([B, c, Hq, d] and [B, Hq, c]); do_chunks the output gradients of those
    rows. Returns three lists (dQ per query chunk, dK and dV per key chunk of
    this rank), in the inputs' dtype. Every rank of `group` calls this with the
    same layout and chunk length.
    """
    import torch
    import torch.distributed as dist

    backward = backward or _fa_backward()
    accumulate = accumulate or _fa_accumulate
    finish = finish or _fa_finish
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if scale is None:
        scale = 1.0 / math.sqrt(q_chunks[0].shape[-1])
    nloc = len(chunk_ids(world, rank, layout))
    for t in (q_chunks, k_chunks, v_chunks, o_chunks, lse_chunks, do_chunks):
        if len(t) != nloc:
            raise ValueError(f"rank {rank} holds {nloc} chunks in the {layout} layout")
    schedule = ring_schedule(world, rank, causal, layout)
    staged = (world > 1 and dist.get_backend(group) == "gloo" and q_chunks[0].is_cuda)
    device = q_chunks[0].device
    acc_dtype = torch.float32 if q_chunks[0].dtype in (torch.bfloat16, torch.float16) \
        else q_chunks[0].dtype

    def wire(t):
        return t.cpu() if staged else t

    def local(t):
        return t.to(device, non_blocking=True) if staged else t

    dq_acc = [torch.zeros(q.shape, dtype=acc_dtype, device=device) for q in q_chunks]
    # one step's per-pair outputs (a step has at most nloc * nloc pairs)
    dq_part = [torch.empty_like(q) for q in q_chunks]
    dk_part = [torch.empty_like(k_chunks[0]) for _ in range(nloc * nloc)]
    dv_part = [torch.empty_like(v_chunks[0]) for _ in range(nloc * nloc)]
    # dK/dV sums of the K/V chunks held at this step: the rank's own at step 0
    acc = ([torch.zeros(k.shape, dtype=acc_dtype, device=device) for k in k_chunks]
           + [torch.zeros(v.shape, dtype=acc_dtype, device=device) for v in v_chunks])
    acc_reqs, sent = [], None
    cur = [wire(t) for t in list(k_chunks) + list(v_chunks)]
    nxt_rank, prv_rank = (rank + 1) % world, (rank - 1) % world
    for step, (src, pairs) in enumerate(schedule):
        kv_reqs, incoming = [], None
        if step + 1 < world:
            incoming = [torch.empty_like(t) for t in cur]
            kv_reqs = _exchange(cur, incoming, nxt_rank, prv_rank, group, _TAG_KV)
        kv = [local(t) for t in cur]
        ks, vs = kv[:nloc], kv[nloc:]
        for j, (qi, ki, m) in enumerate(pairs):
            backward(q_chunks[qi], ks[ki], vs[ki], o_chunks[qi], lse_chunks[qi], do_chunks[qi],
                     m == "causal", scale, dq_part[qi], dk_part[j], dv_part[j])
            accumulate(dq_acc[qi], dq_part[qi])
        # the sums for these K/V chunks, sent by the previous rank after its step
        for r in acc_reqs:
            r.wait()
        acc = [local(t) for t in acc]
        for j, (qi, ki, m) in enumerate(pairs):
            accumulate(acc[ki], dk_part[j])
            accumulate(acc[nloc + ki], dv_part[j])
        if world > 1:
            # on to the rank that holds these chunks next (after the last step: their owner)
            sent = [wire(t) for t in acc]
            acc = [torch.empty_like(t) for t in sent]
            acc_reqs = _exchange(sent, acc, nxt_rank, prv_rank, group, _TAG_ACC)
        for r in kv_reqs:
            r.wait()
        if incoming is not None:
            cur = incoming
    for r in acc_reqs:
        r.wait()
    acc = [local(t) for t in acc]
    dq = [torch.empty_like(q) for q in q_chunks]
    dk = [torch.empty_like(k) for k in k_chunks]
    dv = [torch.empty_like(v) for v in v_chunks]
    for a, out in zip(dq_acc + acc, dq + dk + dv):
        finish(a, out)
    return dq, dk, dv


def _global(rank_in_group, group):
    import torch.distributed as dist
    if group is None:
        return rank_in_group
    return dist.get_global_rank(group, rank_in_group)
