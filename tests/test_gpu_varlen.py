"""GPU parity of the variable-length, paged indexer call (ds4idx_score_topk_varlen) against the
fp64 oracle, sequence by sequence.

Each sequence is an ordinary indexer problem (its own queries, keys, position); the call packs
their queries, stores their keys in one pool (contiguously with gaps, or in shuffled pages) and
scores them in one launch. Every output row must pass the oracle's score / set / order rules
for its own sequence, and the paged and contiguous layouts must give identical outputs.
"""
import numpy as np
import pytest
import torch

from sparse_attention_lightning_indexer_gb300 import ds4idx, inputs

from . import parity

pytestmark = pytest.mark.gpu


def _probs(dtype, shapes, seed):
    return [inputs.make(f"v{b}", T=T, S=S, pos_offset=pos, seed=seed + b, dtype=dtype)
            for b, (T, S, pos) in enumerate(shapes)]


def _pack(probs, dtype, page_size=None, seed=0, gap=37):
    """Packed q/w, and the key pool: contiguous with gaps (page_size None) or shuffled pages."""
    q = torch.cat([p.q for p in probs]).contiguous()
    w = torch.cat([p.w for p in probs]).contiguous()
    cu = [0]
    for p in probs:
        cu.append(cu[-1] + p.T)
    code_dt = probs[0].k.dtype
    if page_size is None:
        starts, rows = [], 0
        for p in probs:
            rows += gap
            starts.append(rows)
            rows += p.S
        rows += gap
        k = torch.zeros((rows, 128), dtype=code_dt)
        ks = torch.zeros(rows, dtype=torch.float32) if dtype == inputs.FP8_E4M3 else None
        for p, s0 in zip(probs, starts):
            k[s0:s0 + p.S] = p.k
            if ks is not None:
                ks[s0:s0 + p.S] = p.kscale
        return q, w, cu, k, ks, starts, None
    n_pages = [(p.S + page_size - 1) // page_size for p in probs]
    total = sum(n_pages) + 3  # a few unused pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(total, generator=g)
    width = max(n_pages) + 2
    table = torch.full((len(probs), width), -1, dtype=torch.int32)
    k = torch.zeros((total * page_size, 128), dtype=code_dt)
    ks = torch.zeros(total * page_size, dtype=torch.float32) if dtype == inputs.FP8_E4M3 else None
    at = 0
    for b, p in enumerate(probs):
        for j in range(n_pages[b]):
            page = int(perm[at])
            at += 1
            table[b, j] = page
            lo, hi = j * page_size, min(p.S, (j + 1) * page_size)
            k[page * page_size:page * page_size + hi - lo] = p.k[lo:hi]
            if ks is not None:
                ks[page * page_size:page * page_size + hi - lo] = p.kscale[lo:hi]
    return q, w, cu, k, ks, None, table


def _run(ix, probs, dtype, page_size=None, seed=0):
    q, w, cu, k, ks, starts, table = _pack(probs, dtype, page_size, seed)
    dev = lambda t: None if t is None else t.cuda()  # noqa: E731
    idx, sc = ix.score_topk_varlen(dev(q), dev(w), cu, dev(k), dev(ks), [p.S for p in probs],
                                   [p.pos_offset for p in probs], kv_start=starts,
                                   page_table=dev(table), page_size=page_size or 0)
    ix.sync_status()
    return idx.cpu().numpy(), sc.cpu().numpy(), cu


def _check(probs, idx, sc, cu):
    for b, p in enumerate(probs):
        if p.T == 0:
            continue
        rows = list(range(p.T))
        parity.check_rows(p, rows, idx[cu[b]:cu[b + 1]], sc[cu[b]:cu[b + 1]])


DECODE_SHAPES = [(1, 9000, 8999), (1, 600, 599), (1, 1, 0), (1, 70000, 69999), (1, 4000, 2500),
                 (1, 513, 512)]
MIXED_SHAPES = [(1, 9000, 8999), (37, 3000, 2963), (0, 500, 0), (300, 2000, 1700), (5, 130, 125),
                (64, 20000, 4000)]


@pytest.mark.parametrize("dtype", [inputs.FP8_E4M3, inputs.BF16])
@pytest.mark.parametrize("shapes", [DECODE_SHAPES, MIXED_SHAPES], ids=["decode", "mixed"])
def test_varlen_contiguous_and_paged(dtype, shapes):
    probs = _probs(dtype, shapes, seed=200)
    with ds4idx.Indexer(dtype, max_T=512, max_S=70000, max_batch=8) as ix:
        i0, s0, cu = _run(ix, probs, dtype)
        _check(probs, i0, s0, cu)
        for page_size in (64, 128, 256):
            i1, s1, _ = _run(ix, probs, dtype, page_size=page_size, seed=page_size)
            assert np.array_equal(i0, i1), page_size
            assert np.array_equal(s0.view(np.uint32), s1.view(np.uint32)), page_size


def test_varlen_matches_the_uniform_batched_call():
    # Equal lengths through the varlen entry (one CTA range per sequence) and the batched entry
    # (sequences interleaved) give the same outputs.
    probs = _probs(inputs.FP8_E4M3, [(1, 40000, 39999 - 977 * b) for b in range(8)], seed=60)
    for p in probs:
        p.pos_offset = 39999 - 977 * probs.index(p)
    with ds4idx.Indexer(inputs.FP8_E4M3, max_T=1, max_S=40000, max_batch=8) as ix:
        q = torch.stack([p.q for p in probs]).cuda()
        w = torch.stack([p.w for p in probs]).cuda()
        k = torch.stack([p.k for p in probs]).cuda()
        ks = torch.stack([p.kscale for p in probs]).cuda()
        ia, sa = ix.score_topk_batched(q, w, k, ks, [p.pos_offset for p in probs])
        ix.sync_status()
        ib, sb, cu = _run(ix, probs, inputs.FP8_E4M3, page_size=128, seed=3)
        assert np.array_equal(ia.cpu().numpy().reshape(8, 512), ib)
        assert np.array_equal(sa.cpu().numpy().reshape(8, 512), sb)
        _check(probs, ib, sb, cu)


def test_varlen_bad_page_ids_are_safe():
    # Page ids past the pool read as zero keys: wrong scores for that sequence, but the call
    # completes and the other sequences are exact.
    dtype = inputs.FP8_E4M3
    probs = _probs(dtype, [(1, 3000, 2999), (1, 2000, 1999)], seed=210)
    q, w, cu, k, ks, _, table = _pack(probs, dtype, 128, seed=1)
    table[1, 3] = 1 << 30
    table[1, 4] = -5
    with ds4idx.Indexer(dtype, max_T=1, max_S=3000, max_batch=2) as ix:
        idx, sc = ix.score_topk_varlen(q.cuda(), w.cuda(), cu, k.cuda(), ks.cuda(), [3000, 2000],
                                       [2999, 1999], page_table=table.cuda(), page_size=128)
        ix.sync_status()
        parity.check_rows(probs[0], [0], idx[:1].cpu().numpy(), sc[:1].cpu().numpy())


def test_varlen_rejects_bad_arguments():
    with ds4idx.Indexer(inputs.BF16, max_T=8, max_S=1000, max_batch=2) as ix:
        q = torch.zeros((3, 64, 128), dtype=torch.bfloat16, device="cuda")
        w = torch.zeros((3, 64), device="cuda")
        k = torch.zeros((256, 128), dtype=torch.bfloat16, device="cuda")
        pt = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
        bad = [
            dict(cu_seqlens_q=[0, 2, 3], kv_start=None, page_table=None),           # neither
            dict(cu_seqlens_q=[0, 2, 3], kv_start=[0, 0], page_table=pt),            # both
            dict(cu_seqlens_q=[1, 2, 3], kv_start=[0, 0], page_table=None),          # cu[0] != 0
            dict(cu_seqlens_q=[0, 3, 2], kv_start=[0, 0], page_table=None),          # decreasing
            dict(cu_seqlens_q=[0, 2, 3], kv_start=[0, 200], page_table=None),        # past pool
            dict(cu_seqlens_q=[0, 2, 3], kv_start=None, page_table=pt, page_size=96),  # page size
            dict(cu_seqlens_q=[0, 2, 3], kv_start=None, page_table=pt, page_size=64,
                 seq_lens=[100, 200]),                                               # table short
        ]
        for kw in bad:
            args = dict(seq_lens=[100, 100], page_size=64 if kw.get("page_table") is not None else 0)
            args.update(kw)
            seq_lens = args.pop("seq_lens")
            with pytest.raises(ds4idx.Ds4IdxError) as e:
                ix.score_topk_varlen(q, w, args.pop("cu_seqlens_q"), k, None, seq_lens, [99, 99],
                                     **args)
            assert e.value.status == ds4idx.ERR_INVALID_ARG, kw
