"""Context-parallel (ring) attention across ranks.

The FlexAttention page lists context parallelism among the variants it
composes with sliding window, document masking and causal masks, and the
Online-Softmax/FlashAttention page names FlashAttention in distributed
training and inference. This module is the host-side schedule of that
composition: a sequence of S positions is cut into ``world`` contiguous
shards; rank r holds query shard r and key/value shard r. For N = world
steps each rank attends its queries to the key/value shard it currently
holds (one forward call with the shards' absolute position offsets, so every
mask term, ALiBi and the document ids see whole-sequence positions), passes
that shard to rank r + 1 and receives the next one from rank r - 1. The
exchange of step s overlaps the compute of step s. After N steps every rank
has seen every key/value shard, and the partial results merge by the
online-softmax merge (``attn_combine``):

    LSE = ln sum_k e^(LSE_k),    O = sum_k e^(LSE_k - LSE) O_k

A (query shard, key shard) pair that the mask provably empties (a key shard
wholly after the query shard under a causal mask, or wholly outside the
sliding window, and wholly past every prefix) is not computed.

The per-shard compute and the merge are parameters: on GPUs they are the
library's ``attn_fwd`` and ``attn_combine`` (``library_shard_forward``,
``library_merge``), with the exchange over NCCL; the CPU tests pass other
implementations of the same two steps and exchange over gloo.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

__all__ = ["shard_cuts", "pair_may_keep", "ring_order", "ring_forward",
           "library_shard_forward", "library_merge"]


def shard_cuts(S: int, world: int) -> List[int]:
    """Cut points of ``world`` contiguous shards of S positions, as even as
    possible (the first S % world shards are one longer): shard r covers
    positions cuts[r] .. cuts[r + 1] - 1."""
    if world < 1 or S < 0:
        raise ValueError("shard_cuts: world >= 1 and S >= 0")
    base, extra = divmod(S, world)
    cuts = [0]
    for r in range(world):
        cuts.append(cuts[-1] + base + (1 if r < extra else 0))
    return cuts


def pair_may_keep(causal: bool, window: int, prefix_max: Optional[int], q_lo: int, q_hi: int,
                  kv_lo: int, kv_hi: int) -> bool:
    """False only when no (query, key) pair of absolute positions
    q_lo <= i < q_hi, kv_lo <= j < kv_hi can be kept by the mask
    ``(causal AND window AND document) OR prefix``: the AND-terms exclude
    every pair (keys all after the last query under causal, or all at least
    ``window`` behind the first query) and no key lies inside the longest
    prefix ``prefix_max`` (None: no prefix term). The document term is never
    used to exclude a pair (it would need the ids)."""
    if q_hi <= q_lo or kv_hi <= kv_lo:
        return False
    and_part = True
    if causal and kv_lo > q_hi - 1:
        and_part = False
    if window and window > 0 and q_lo - (kv_hi - 1) >= window:
        and_part = False
    prefix_part = prefix_max is not None and kv_lo < prefix_max
    return and_part or prefix_part


def ring_order(rank: int, world: int) -> List[int]:
    """Key/value shard held by ``rank`` at each step: its own first, then
    the shards passed along the ring, (rank - s) mod world at step s."""
    return [(rank - s) % world for s in range(world)]


def _exchange(k_cur, v_cur, k_buf, v_buf, rank: int, world: int, group):
    """Starts sending the held shard to rank + 1 and receiving the next one
    from rank - 1; returns the requests to wait on."""
    import torch.distributed as dist
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    ops = [dist.P2POp(dist.isend, k_cur, nxt, group), dist.P2POp(dist.isend, v_cur, nxt, group),
           dist.P2POp(dist.irecv, k_buf, prv, group), dist.P2POp(dist.irecv, v_buf, prv, group)]
    return dist.batch_isend_irecv(ops)


def ring_forward(q, k, v, *, rank: int, world: int, cuts: Sequence[int],
                 shard_forward: Callable, merge: Callable, causal: bool = False,
                 window: int = 0, prefix_max: Optional[int] = None, group=None,
                 trace: Optional[list] = None) -> Tuple[object, object]:
    """Ring attention for this rank's shards.

    ``q`` [B, Hq, Sq_r, D] is query shard ``rank`` and ``k``/``v``
    [B, Hkv, Skv_r, D] key/value shard ``rank`` (torch tensors, contiguous),
    the shards of positions cuts[rank] .. cuts[rank + 1] - 1 of one sequence.
    ``shard_forward(q, k, v, q_offset, kv_offset)`` returns the partial
    ``(O, LSE)`` of the queries against one key/value shard at those absolute
    offsets; ``merge(parts)`` merges a list of them. ``causal``, ``window``
    and ``prefix_max`` (the largest prefix length, or None) describe the mask
    only so that provably empty pairs are skipped. Ranks exchange shards
    with torch.distributed point-to-point calls on ``group``. ``trace``
    (optional list) receives the (step, key shard, computed) triples.
    Returns the merged ``(O, LSE)`` of the queries over the whole sequence."""
    import torch
    if len(cuts) != world + 1:
        raise ValueError("ring_forward: cuts must hold world + 1 cut points")
    order = ring_order(rank, world)
    q_lo, q_hi = cuts[rank], cuts[rank + 1]
    k_cur, v_cur = k, v
    parts = []
    for s, j in enumerate(order):
        reqs = None
        if s + 1 < world:
            nj = order[s + 1]  # the shard rank - 1 holds now
            n = cuts[nj + 1] - cuts[nj]
            k_buf = torch.empty((k.shape[0], k.shape[1], n, k.shape[3]), dtype=k.dtype,
                                device=k.device)
            v_buf = torch.empty((v.shape[0], v.shape[1], n, v.shape[3]), dtype=v.dtype,
                                device=v.device)
            reqs = _exchange(k_cur, v_cur, k_buf, v_buf, rank, world, group)
        kv_lo, kv_hi = cuts[j], cuts[j + 1]
        run = j == rank or pair_may_keep(causal, window, prefix_max, q_lo, q_hi, kv_lo, kv_hi)
        if run:
            parts.append(shard_forward(q, k_cur, v_cur, q_lo, kv_lo))
        if trace is not None:
            trace.append((s, j, run))
        if reqs is not None:
            for r in reqs:
                r.wait()
            k_cur, v_cur = k_buf, v_buf
    return merge(parts)


def library_shard_forward(variant: int, *, window: int = 0, softcap: float = 0.0,
                          doc_id=None, prefix_len=None, alibi_slopes=None,
                          scale: float = 0.0, stream=None) -> Callable:
    """The per-shard compute on the GPU: builds the block mask of the shard
    pair with its offsets and runs ``attn_fwd`` into new output tensors.
    ``doc_id`` covers the whole sequence ([B, S], absolute positions)."""
    import torch
    import masked_attention_gb300 as M

    def run(q, k, v, q_offset: int, kv_offset: int):
        B, Hq, Sq, _ = q.shape
        Skv = k.shape[2]
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
        bm = None
        if variant & 0xF:
            bm = M.build_block_mask(variant & 0xF, B, Sq, Skv, window=window, doc_id=doc_id,
                                    prefix_len=prefix_len, q_offset=q_offset,
                                    kv_offset=kv_offset, device=q.device, stream=stream)
        M.attn_fwd(q, k, v, o, lse, variant, window=window, softcap=softcap, doc_id=doc_id,
                   prefix_len=prefix_len, alibi_slopes=alibi_slopes, scale=scale,
                   block_mask=bm, q_offset=q_offset, kv_offset=kv_offset, stream=stream)
        return o, lse

    return run


def library_merge(parts, stream=None):
    """The merge on the GPU: ``attn_combine`` over the partial results."""
    import torch
    import masked_attention_gb300 as M
    o_parts = torch.stack([o for o, _ in parts]).contiguous()
    l_parts = torch.stack([l for _, l in parts]).contiguous()
    o = torch.empty_like(parts[0][0])
    lse = torch.empty_like(parts[0][1])
    M.attn_combine(o_parts, l_parts, o, lse, stream=stream)
    return o, lse
