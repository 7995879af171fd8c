"""Context parallelism over ranks: the bookkeeping that turns one global batch
into each rank's local call, and the exchange that joins partial results.

Two ways of cutting a long context across ranks, both from the pages:

* Query split ("sparse_flash_mla", CP example: two CP ranks run one after
  the other in a single process).  The global TND query tokens are cut into
  contiguous ranges, one per rank.  A rank passes only its own query rows,
  and for each sequence the KV length up to the end of those rows, so that the
  kernels' right-down alignment (row i at p = kv_len - q_len + i) puts the
  rank's first row exactly at the cut.  Every output row is computed by one
  rank; nothing needs combining.
* KV split (the ring-attention use of softmax_lse, "aclnnFusedInferAttention-
  ScoreV2").  Each sequence's keys are cut at block boundaries into one part
  per rank; every rank computes all query rows against its part and returns
  (out, lse); the parts are joined with the log-sum-exp combine
  (fia_lse_combine).  A sink must enter once: the parts run without sinks
  and the combine adds them.

The functions here only compute lengths, tables and ranges (host integers and
small tensors); the attention itself runs in libfia's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import torch


@dataclasses.dataclass
class QuerySlice:
    """One rank's part of a query split."""
    token_begin: int            # first global query token of the rank
    token_end: int              # one past the last
    batches: List[int]          # global sequence of each local batch
    q_lens: List[int]           # local query rows of each local batch
    kv_lens: List[int]          # KV prefix each local batch passes (seqused_kv)
    row_begin: List[int]        # first row of each local batch within its sequence

    @property
    def cu_seqlens_q(self) -> List[int]:
        out = [0]
        for q in self.q_lens:
            out.append(out[-1] + q)
        return out


def query_split(cu_seqlens_q: Sequence[int], kv_lens: Sequence[int], world: int,
                rank: int) -> QuerySlice:
    """Rank `rank` of `world` takes global query tokens [T*rank/world,
    T*(rank+1)/world).  For each sequence it overlaps, rows s..e-1 of the
    sequence, it passes q_len = e - s and the KV prefix kv_len - q_len_global
    + e: the keys up to its last row's position.  Right-down alignment then
    gives row s + i' the position it has in the whole call."""
    T = cu_seqlens_q[-1]
    lo, hi = T * rank // world, T * (rank + 1) // world
    batches, qls, kvs, rows = [], [], [], []
    for b in range(len(kv_lens)):
        t0, t1 = cu_seqlens_q[b], cu_seqlens_q[b + 1]
        s, e = max(t0, lo), min(t1, hi)
        if s >= e:
            continue
        ql_global = t1 - t0
        batches.append(b)
        qls.append(e - s)
        kvs.append(kv_lens[b] - ql_global + (e - t0))
        rows.append(s - t0)
    return QuerySlice(lo, hi, batches, qls, kvs, rows)


@dataclasses.dataclass
class KvSlice:
    """One rank's part of a KV split."""
    block_table: torch.Tensor   # int32 [B, max local blocks]
    kv_lens: List[int]          # keys of each sequence in this part (run without sinks)


def kv_split(block_table: torch.Tensor, kv_lens: Sequence[int], block_size: int, world: int,
             rank: int) -> KvSlice:
    """Rank `rank` of `world` takes blocks [n*rank/world, n*(rank+1)/world) of
    each sequence's n = ceil(kv_len / block_size) blocks (whole blocks, so the
    pages need no copying): its table lists those block ids, its length is
    the number of keys they hold.  Positions inside a part start again at 0,
    so this split is for calls in which every query row sees every key of its
    sequence: mask mode 0, or one query row per sequence under a causal
    mask (decode)."""
    B = len(kv_lens)
    parts, lens = [], []
    for b in range(B):
        n = -(-kv_lens[b] // block_size)
        b0, b1 = n * rank // world, n * (rank + 1) // world
        parts.append(block_table[b, b0:b1])
        lens.append(max(0, min(kv_lens[b], b1 * block_size) - b0 * block_size))
    width = max(1, max(p.numel() for p in parts))
    spare = block_table.reshape(-1)[:1].expand(width)
    table = torch.stack([torch.cat([p, spare[p.numel():]]) for p in parts]).to(torch.int32)
    return KvSlice(table.contiguous(), lens)


def gather_parts(out: torch.Tensor, lse: torch.Tensor, group=None):
    """All-gather every rank's (out, lse) of a KV split: lists ordered by rank,
    ready for the combine (fia_lse_combine on the GPU)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    outs = [torch.empty_like(out) for _ in range(world)]
    lses = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(outs, out.contiguous(), group=group)
    dist.all_gather(lses, lse.contiguous(), group=group)
    return outs, lses
