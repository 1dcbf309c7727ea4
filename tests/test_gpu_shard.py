"""GPU checks of the sharded indexer's compute pieces on one GPU: the merge kernel
(ds4idx_merge_topk) against the oracle, and key-range and query-row sharding emulated rank by
rank on one device, whose results must equal the unsharded call bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_attention_lightning_indexer_gb300 import ds4idx, inputs, shard

from . import parity

pytestmark = pytest.mark.gpu


def test_merge_matches_the_oracle_selection():
    # Random disjoint lists with ties across lists, empty slots, and a list with no rows at first.
    rng = np.random.default_rng(4)
    L, rows = 5, 37
    offs = [0, 700, 1400, 2100, 2800]
    row0 = [0, 0, 3, 0, 10]
    idx = np.full((L, rows, 512), -1, dtype=np.int32)
    sc = np.full((L, rows, 512), -np.inf, dtype=np.float32)
    for l in range(L):
        for r in range(row0[l], rows):
            n = rng.integers(0, 513)
            keys = rng.choice(700, size=n, replace=False)
            vals = rng.choice(np.float32([-1.5, 0.0, 0.25, 3.0]), size=n).astype(np.float32)
            vals += (rng.integers(0, 3, size=n) * 0.5).astype(np.float32)
            idx[l, r, :n], sc[l, r, :n] = keys, vals
    gi, gs = ds4idx.merge_topk(torch.from_numpy(idx).cuda(), torch.from_numpy(sc).cuda(), offs, row0)
    torch.cuda.synchronize()
    full = np.full((rows, 3500), -np.inf, dtype=np.float32)
    for l in range(L):
        for r in range(row0[l], rows):
            m = idx[l, r] >= 0
            full[r, idx[l, r][m] + offs[l]] = sc[l, r][m]
    # every key present is "visible"; -inf marks absent keys, which the selection never keeps
    # ahead of a present one (present scores are finite)
    want_i, want_s = orc.select(full, np.full(rows, 3500), 512)
    present = np.isfinite(full).sum(axis=1)
    for r in range(rows):
        m = min(512, present[r])
        assert np.array_equal(gi[r, :m].cpu().numpy(), want_i[r, :m]), r
        assert np.array_equal(gs[r, :m].cpu().numpy(), want_s[r, :m]), r
        assert np.all(gi[r, m:].cpu().numpy() == -1)


@pytest.mark.parametrize("dtype", [inputs.FP8_E4M3, inputs.BF16])
@pytest.mark.parametrize("T,S,pos,world", [(1, 40000, 39999, 3), (300, 6000, 5700, 4),
                                           (64, 3000, 200, 2)])
def test_key_sharded_equals_unsharded(dtype, T, S, pos, world):
    prob = inputs.make("ks", T=T, S=S, pos_offset=pos, seed=230 + T, dtype=dtype)
    q, w, k, ks = parity.to_device(prob)
    with ds4idx.Indexer(dtype, max_T=T, max_S=S) as ix:
        ref_i, ref_s = ix.score_topk(q, w, k, ks, pos)
        lists_i, lists_s, offs, firsts = [], [], [], []
        for r in range(world):  # each "rank" in turn, on this one GPU
            s0, s1 = shard.key_range(S, world, r)
            li = torch.empty((T, 512), dtype=torch.int32, device="cuda")
            ls = torch.empty((T, 512), dtype=torch.float32, device="cuda")
            tf = shard.first_visible_row(pos, s0) if s1 > s0 else T
            if tf < T:
                ix.score_topk(q[tf:], w[tf:], k[s0:s1], None if ks is None else ks[s0:s1],
                              pos + tf - s0, out_idx=li[tf:], out_score=ls[tf:])
            lists_i.append(li)
            lists_s.append(ls)
            offs.append(s0)
            firsts.append(tf)
        gi, gs = ds4idx.merge_topk(torch.stack(lists_i), torch.stack(lists_s), offs, firsts)
        ix.sync_status()
    assert torch.equal(gi, ref_i)
    assert torch.equal(gs, ref_s)
    parity.check_rows(prob, list(range(T)), gi.cpu().numpy(), gs.cpu().numpy())


@pytest.mark.parametrize("world", [2, 3])
def test_row_sharded_equals_unsharded(world):
    prob = inputs.make("rs", T=2000, S=2000, pos_offset=0, seed=240, dtype=inputs.BF16)
    q, w, k, _ = parity.to_device(prob)
    with ds4idx.Indexer(prob.dtype, max_T=prob.T, max_S=prob.S) as ix:
        ref_i, ref_s = ix.score_topk(q, w, k, None, 0)
        oi = torch.full_like(ref_i, -7)
        os_ = torch.full_like(ref_s, 7.0)
        for r in range(world):
            shard.score_topk_row_sharded(ix, q, w, k, None, 0, r, world, oi, os_)
        ix.sync_status()
    assert torch.equal(oi, ref_i) and torch.equal(os_, ref_s)
