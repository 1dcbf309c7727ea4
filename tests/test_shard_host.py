"""Host logic of the sharded indexer (sparse_attention_lightning_indexer_gb300/shard.py) on CPU:
the row and key plans, and the key-range exchange with two gloo ranks.

The exchange test checks the property the key-sharded call rests on, with the oracle standing in
for each rank's GPU scoring (test infrastructure only): the Top-512 of the union of the ranks'
per-range Top-512 lists, gathered through torch.distributed, is the oracle's global Top-512.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_attention_lightning_indexer_gb300 import inputs, shard


@pytest.mark.parametrize("T,world", [(65536, 2), (65536, 8), (1001, 3), (7, 4), (4, 2)])
def test_zigzag_rows_cover_once_and_balance(T, world):
    seen = np.zeros(T, dtype=int)
    work = []
    for r in range(world):
        chunks = shard.zigzag_row_chunks(T, world, r)
        for a, b in chunks:
            assert a % 4 == 0 and a < b <= T
            seen[a:b] += 1
        work.append(sum(shard.causal_pairs(0, T, a, b) for a, b in chunks))
    assert np.all(seen == 1)
    if T >= 1024:
        # zig-zag pairs a short chunk with a long one: every rank within 1% of the mean work
        assert max(work) / (sum(work) / world) < 1.01
        # contiguous shares would be far off (the last rank does 1.5x (W = 2) to ~2x the mean)
        share = T // world
        last = shard.causal_pairs(0, T, T - share, T)
        assert last / (sum(work) / world) > 1.45


@pytest.mark.parametrize("S,world", [(262144, 2), (262144, 8), (1000, 3), (129, 4), (1, 2)])
def test_key_ranges_tile_the_cache(S, world):
    prev = 0
    for r in range(world):
        s0, s1 = shard.key_range(S, world, r)
        assert s0 == prev and s0 <= s1 <= S
        assert s0 % 128 == 0
        prev = s1
    assert prev == S


def test_first_visible_row():
    assert shard.first_visible_row(260096, 0) == 0
    assert shard.first_visible_row(260096, 131072) == 0
    assert shard.first_visible_row(100, 228) == 128
    assert shard.first_visible_row(0, 512) == 512


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import oracle as orc
    prob = inputs.make("ks", T=6, S=3000, pos_offset=2994, seed=7, dtype=inputs.BF16)
    q, k = prob.codes()
    s0, s1 = shard.key_range(prob.S, world, rank)
    t_first = shard.first_visible_row(prob.pos_offset, s0)
    # this rank's lists: the oracle's Top-512 of its key range (rows before t_first stay empty)
    idx = np.full((prob.T, 512), -1, dtype=np.int32)
    sc = np.full((prob.T, 512), -np.inf, dtype=np.float32)
    if t_first < prob.T:
        rows = np.arange(t_first, prob.T)
        i, v = orc.topk(prob.dtype, q[t_first:], prob.w.numpy()[t_first:], k[s0:s1], None,
                        prob.pos_offset + t_first - s0, 512)
        idx[rows], sc[rows] = i, v.astype(np.float32)
    all_idx, all_sc = shard.exchange_lists(torch.from_numpy(idx), torch.from_numpy(sc))
    starts = [None] * world
    dist.all_gather_object(starts, (s0, t_first))
    if rank == 0:
        # the union of the gathered lists, with global indices, reselected by the oracle
        n_vis = np.array([prob.n_visible(t) for t in range(prob.T)])
        full = np.full((prob.T, prob.S), -np.inf)
        for r, (a, tf) in enumerate(starts):
            for t in range(tf, prob.T):
                for j, v in zip(all_idx[r, t].tolist(), all_sc[r, t].tolist()):
                    if j >= 0:
                        full[t, a + j] = v
        # keys not in any list score -inf; the set must still be the global Top-512
        got, _ = orc.select(full, n_vis, 512)
        want, _ = orc.topk(prob.dtype, q, prob.w.numpy(), k, None, prob.pos_offset, 512)
        out["ok"] = bool(np.array_equal(got, want))
        out["starts"] = starts
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_key_shards_union_holds_the_global_top512():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res["starts"] == [(0, 0), (1536, 0)]
    assert res["ok"]
