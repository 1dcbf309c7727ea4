"""Sharding the indexer over several processes (one GPU each): the plans, the exchange and the
sharded calls. Every score and every selection runs in the library's kernels; this module
decides which rows or keys each rank takes, moves the per-rank lists with torch.distributed and
calls the library's merge.

Two ways to split one indexer call (the pages describe single-device engines; these are the
plain ways to spread the same computation):
  * query rows (long prefills): rows are independent, so each rank scores a share of the queries
    against all visible keys and no exchange is needed. A causal row t costs about t + 1 keys,
    so contiguous equal shares are unequal work; the rows are cut into 2 * world chunks and rank
    r takes chunks r and 2 * world - 1 - r (a short and a long one), which balances the causal
    triangle to within one chunk.
  * key ranges (long caches, decode): each rank scores all queries against a contiguous range of
    the keys and keeps that range's Top-512; the union of the ranks' lists holds the global
    Top-512 (a key among the best 512 of all keys is among the best 512 of its range), so an
    all-gather of the lists and one merge (ds4idx_merge_topk) finish the call. Query t sees none
    of range [s0, s1) when pos_offset + t < s0: such rows are left out of that rank's call and
    marked empty for the merge.
"""
from __future__ import annotations

import torch

from . import ds4idx

TILE = 128  # keys per tile of the indexer kernel: key ranges are cut on tile boundaries


def zigzag_row_chunks(T: int, world: int, rank: int) -> list[tuple[int, int]]:
    """The query-row chunks [t0, t1) of rank `rank`: chunks r and 2W-1-r of 2W near-equal
    chunks (4-query aligned, empty chunks dropped)."""
    if world < 1 or not 0 <= rank < world or T < 0:
        raise ValueError("bad world/rank/T")
    n = 2 * world
    blocks = (T + 3) // 4
    bounds = [min(T, 4 * ((blocks * i) // n)) for i in range(n + 1)]
    out = []
    for c in (rank, n - 1 - rank):
        if bounds[c] < bounds[c + 1]:
            out.append((bounds[c], bounds[c + 1]))
    return out


def causal_pairs(pos_offset: int, S: int, t0: int, t1: int) -> int:
    """Visible (query, key) pairs of rows t0..t1-1 (the work of a row chunk)."""
    return sum(min(pos_offset + t, S - 1) + 1 for t in range(t0, t1))


def key_range(S: int, world: int, rank: int) -> tuple[int, int]:
    """Rank `rank`'s contiguous key range [s0, s1), cut on 128-key tile boundaries."""
    if world < 1 or not 0 <= rank < world or S < 1:
        raise ValueError("bad world/rank/S")
    tiles = (S + TILE - 1) // TILE
    s0 = min(S, TILE * ((tiles * rank) // world))
    s1 = min(S, TILE * ((tiles * (rank + 1)) // world))
    return s0, s1


def first_visible_row(pos_offset: int, s0: int) -> int:
    """First query row that sees key s0 (rows before it see none of a range starting at s0)."""
    return max(0, s0 - pos_offset)


def exchange_lists(idx: torch.Tensor, score: torch.Tensor, group=None):
    """All-gather of every rank's [rows, 512] lists: returns ([W, rows, 512], [W, rows, 512]).
    With NCCL the tensors stay on the GPU; with gloo they move through host memory."""
    world = torch.distributed.get_world_size(group)
    all_idx = [torch.empty_like(idx) for _ in range(world)]
    all_sc = [torch.empty_like(score) for _ in range(world)]
    torch.distributed.all_gather(all_idx, idx.contiguous(), group=group)
    torch.distributed.all_gather(all_sc, score.contiguous(), group=group)
    return torch.stack(all_idx), torch.stack(all_sc)


def score_topk_row_sharded(ix: ds4idx.Indexer, q, w, kcache, kscale, pos_offset: int,
                           rank: int, world: int, out_idx=None, out_score=None):
    """This rank's share of a query-row-sharded call: each of its zig-zag chunks [a, b) is one
    indexer call on rows a..b-1 at position pos_offset + a, written into rows a..b-1 of
    out_idx / out_score ([T, 512], allocated when not given; other rows are left untouched).
    Returns (chunks, out_idx, out_score)."""
    T = q.shape[0]
    dev = q.device
    if out_idx is None:
        out_idx = torch.empty((T, ds4idx.TOPK), dtype=torch.int32, device=dev)
    if out_score is None:
        out_score = torch.empty((T, ds4idx.TOPK), dtype=torch.float32, device=dev)
    chunks = zigzag_row_chunks(T, world, rank)
    for a, b in chunks:
        ix.score_topk(q[a:b], w[a:b], kcache, kscale, pos_offset + a, out_idx=out_idx[a:b],
                      out_score=out_score[a:b])
    return chunks, out_idx, out_score


def score_topk_key_sharded(ix: ds4idx.Indexer, q, w, kcache_range, kscale_range, s0: int,
                           pos_offset: int, group=None):
    """A key-range-sharded call: this rank holds keys [s0, s0 + len) of the cache and every rank
    holds all T queries. Each rank scores its range, the lists are all-gathered and merged.
    Returns the global (idx [T, 512], score [T, 512]) on every rank."""
    T = q.shape[0]
    dev = q.device
    # rows before t_first are never read: the merge is told that this list starts there
    idx = torch.empty((T, ds4idx.TOPK), dtype=torch.int32, device=dev)
    sc = torch.empty((T, ds4idx.TOPK), dtype=torch.float32, device=dev)
    t_first = first_visible_row(pos_offset, s0) if kcache_range.shape[0] > 0 else T
    if t_first < T:
        ix.score_topk(q[t_first:], w[t_first:], kcache_range, kscale_range,
                      pos_offset + t_first - s0, out_idx=idx[t_first:], out_score=sc[t_first:])
    all_idx, all_sc = exchange_lists(idx, sc, group)
    world = all_idx.shape[0]
    starts = [None] * world
    torch.distributed.all_gather_object(starts, (int(s0), int(t_first)), group=group)
    return ds4idx.merge_topk(all_idx, all_sc, [a for a, _ in starts], [b for _, b in starts])
