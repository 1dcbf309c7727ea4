"""GPU parity: the CUDA indexer (through the C ABI) against the fp64 oracle.

Sizes here are ones the oracle finishes in seconds while still spanning several 128-key tiles,
several 4-query blocks, ragged tails of both, key-range splits and the merge kernel. Every row
is checked with the score / set / order rules and the selection rerun on the kernel's own fp32
scores (tests/parity.py).
"""
import numpy as np
import pytest
import torch

from sparse_attention_lightning_indexer_gb300 import inputs
from sparse_attention_lightning_indexer_gb300 import ds4idx

from . import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bf16_ix():
    with ds4idx.Indexer(ds4idx.BF16, max_T=16384, max_S=65536, max_batch=8) as ix:
        yield ix


@pytest.fixture(scope="module")
def fp8_ix():
    with ds4idx.Indexer(ds4idx.FP8_E4M3, max_T=16384, max_S=65536, max_batch=8) as ix:
        yield ix


def _ix(prob, bf16_ix, fp8_ix):
    return bf16_ix if prob.dtype == inputs.BF16 else fp8_ix


def run_full(prob, ix, rerun=True):
    dev = parity.to_device(prob)
    idx, sc = ix.score_topk(*dev, pos_offset=prob.pos_offset)
    ix.sync_status()
    rows = list(range(prob.T))
    gi, gs = idx.cpu().numpy(), sc.cpu().numpy()
    stats = parity.check_rows(prob, rows, gi, gs)
    if rerun:
        dense = ix.score_dense_debug(*dev, pos_offset=prob.pos_offset).cpu().numpy()
        parity.rerun_selection(prob, rows, dense, gi, gs)
    return stats, gi, gs


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.FP8_E4M3])
def test_ragged_prefill(dtype, bf16_ix, fp8_ix):
    # T = S = 1001: 8 key tiles with a 105-key tail, 251 query blocks with a 1-query tail.
    prob = inputs.make("ragged", T=1001, S=1001, pos_offset=0, seed=11, dtype=dtype)
    stats, _, _ = run_full(prob, _ix(prob, bf16_ix, fp8_ix))
    assert stats["rows"] == 1001


def test_tiny_1k_workload(bf16_ix):
    prob = inputs.workload("tiny_1k")
    stats, gi, _ = run_full(prob, bf16_ix)
    # Rows with at most 512 visible keys keep all of them.
    for t in range(512):
        assert sorted(gi[t, :t + 1].tolist()) == list(range(t + 1))


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.FP8_E4M3])
def test_pos_offset_chunk(dtype, bf16_ix, fp8_ix):
    # A 300-token chunk at position 1700 of a 2000-key cache (chunked prefill).
    prob = inputs.make("chunk", T=300, S=2000, pos_offset=1700, seed=12, dtype=dtype)
    run_full(prob, _ix(prob, bf16_ix, fp8_ix))


@pytest.mark.parametrize("pos", [506, 507, 508, 509])
def test_visible_count_around_512(pos, bf16_ix):
    # Rows see 507..516 keys: fewer than, exactly and just over 512.
    prob = inputs.make("edge512", T=7, S=700, pos_offset=pos, seed=13, dtype=inputs.BF16)
    stats, gi, _ = run_full(prob, bf16_ix)
    for t in range(7):
        n = prob.n_visible(t)
        if n <= 512:
            assert sorted(gi[t, :n].tolist()) == list(range(n))


def test_single_query_split_merge(bf16_ix, fp8_ix):
    # T = 1 takes the one-query kernel with the key range split over many CTAs + merge kernel.
    for dtype, ix in ((inputs.BF16, bf16_ix), (inputs.FP8_E4M3, fp8_ix)):
        prob = inputs.make("decode1", T=1, S=9000, pos_offset=8999, seed=14, dtype=dtype)
        run_full(prob, ix)


def test_batched_decode_small(fp8_ix):
    probs = [inputs.make(f"b{b}", T=1, S=6000, pos_offset=p, seed=20 + b,
                         dtype=inputs.FP8_E4M3)
             for b, p in enumerate((5999, 3000, 10, 511))]
    q = torch.stack([p.q for p in probs]).cuda()
    w = torch.stack([p.w for p in probs]).cuda()
    k = torch.stack([p.k for p in probs]).cuda()
    ks = torch.stack([p.kscale for p in probs]).cuda()
    idx, sc = fp8_ix.score_topk_batched(q, w, k, ks, [p.pos_offset for p in probs])
    fp8_ix.sync_status()
    for b, prob in enumerate(probs):
        parity.check_rows(prob, [0], idx[b].cpu().numpy(), sc[b].cpu().numpy())


def test_batched_chunk_bf16(bf16_ix):
    probs = [inputs.make(f"c{b}", T=37, S=3000, pos_offset=p, seed=30 + b, dtype=inputs.BF16)
             for b, p in enumerate((2963, 100, 0))]
    q = torch.stack([p.q for p in probs]).cuda()
    w = torch.stack([p.w for p in probs]).cuda()
    k = torch.stack([p.k for p in probs]).cuda()
    idx, sc = bf16_ix.score_topk_batched(q, w, k, None, [p.pos_offset for p in probs])
    bf16_ix.sync_status()
    for b, prob in enumerate(probs):
        parity.check_rows(prob, list(range(37)), idx[b].cpu().numpy(), sc[b].cpu().numpy())


def test_tie_storm_lowest_indices(bf16_ix):
    # k = 0: every score is exactly 0, so each row must return its lowest min(512, n) keys.
    prob = inputs.make("ties", T=64, S=2000, pos_offset=1000, seed=15, dtype=inputs.BF16)
    prob.k.zero_()
    stats, gi, gs = run_full(prob, bf16_ix)
    for t in range(64):
        assert gi[t].tolist() == list(range(512))
        assert np.all(gs[t] == 0.0)


def test_all_negative_scores(bf16_ix):
    prob = inputs.make("neg", T=50, S=1500, pos_offset=1400, seed=16, dtype=inputs.BF16)
    prob.w.copy_(-prob.w.abs())
    stats, _, gs = run_full(prob, bf16_ix)
    assert np.all(gs[np.isfinite(gs)] <= 0.0)


def test_zero_key_scales(fp8_ix):
    prob = inputs.make("kscale0", T=40, S=1200, pos_offset=1100, seed=17, dtype=inputs.FP8_E4M3)
    prob.kscale[::3] = 0.0
    run_full(prob, fp8_ix)


def test_deterministic(bf16_ix):
    prob = inputs.make("det", T=257, S=3000, pos_offset=2743, seed=18, dtype=inputs.BF16)
    dev = parity.to_device(prob)
    a = [t.clone() for t in bf16_ix.score_topk(*dev, pos_offset=prob.pos_offset)]
    b = bf16_ix.score_topk(*dev, pos_offset=prob.pos_offset)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0])
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


def test_invalid_arguments_rejected(bf16_ix, fp8_ix):
    lib = ds4idx.load()
    prob = inputs.make("args", T=8, S=64, pos_offset=0, seed=19, dtype=inputs.BF16)
    q, w, k, _ = parity.to_device(prob)
    oi = torch.empty((8, 512), dtype=torch.int32, device="cuda")
    os_ = torch.empty((8, 512), dtype=torch.float32, device="cuda")
    h = bf16_ix.handle
    P = lambda t: t.data_ptr()  # noqa: E731
    s = torch.cuda.current_stream().cuda_stream
    ok = lib.ds4idx_score_topk(h, P(q), P(w), P(k), None, 8, 64, 0, 512, P(oi), P(os_), s)
    assert ok == ds4idx.OK
    cases = [
        (None, P(w), P(k), None, 8, 64, 0, 512),            # null q
        (P(q) + 2, P(w), P(k), None, 8, 64, 0, 512),        # misaligned q
        (P(q), P(w), P(k), P(w), 8, 64, 0, 512),            # kscale given for bf16
        (P(q), P(w), P(k), None, 8, 64, 0, 256),            # topk mismatch
        (P(q), P(w), P(k), None, 8, 0, 0, 512),             # S = 0
        (P(q), P(w), P(k), None, 8, 64, -1, 512),           # negative position
        (P(q), P(w), P(k), None, 20000, 64, 0, 512),        # T > max_T
        (P(q), P(w), P(k), None, 8, 1 << 20, 0, 512),       # S > max_S
    ]
    for c in cases:
        st = lib.ds4idx_score_topk(h, *c, P(oi), P(os_), s)
        assert st == ds4idx.ERR_INVALID_ARG, c
    assert lib.ds4idx_score_topk(h, P(q), P(w), P(k), None, 8, 64, 0, 512, None, None, s) \
        == ds4idx.ERR_INVALID_ARG
    # FP8 handle without kscale
    assert lib.ds4idx_score_topk(fp8_ix.handle, P(q), P(w), P(k), None, 8, 64, 0, 512, P(oi),
                                 P(os_), s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_score_topk(None, P(q), P(w), P(k), None, 8, 64, 0, 512, P(oi), P(os_),
                                 s) == ds4idx.ERR_INVALID_ARG
    # T = 0 is a no-op
    assert lib.ds4idx_score_topk(h, P(q), P(w), P(k), None, 0, 64, 0, 512, P(oi), P(os_),
                                 s) == ds4idx.OK
    bf16_ix.sync_status()


def test_unsupported_config():
    with pytest.raises(ds4idx.Ds4IdxError) as e:
        ds4idx.Indexer(ds4idx.BF16, max_T=16, max_S=16, n_heads=32)
    assert e.value.status == ds4idx.ERR_UNSUPPORTED


def test_split_merge_concentrated_winners(fp8_ix, bf16_ix):
    # 400 consecutive keys aligned with every query dominate the Top-512, so one or two key
    # splits hold most of it: the prefix path of the split merge must see that its 64-word
    # prefixes are not enough and fall back to the full merge.
    for dtype, ix in ((inputs.FP8_E4M3, fp8_ix), (inputs.BF16, bf16_ix)):
        prob = inputs.make("hot", T=1, S=30000, pos_offset=29999, seed=21, dtype=dtype)
        prob.w.copy_(prob.w.abs())
        if dtype == inputs.BF16:
            prob.q.copy_(prob.q.abs())
            prob.k[12000:12400] = (prob.k[12000:12400].float().abs() * 3.0).to(torch.bfloat16)
        else:
            prob.q.bitwise_and_(0x7F)  # clear E4M3 sign bits: |q|
            prob.k[12000:12400] = prob.k[12000:12400].bitwise_and(0x7F)
            prob.kscale[12000:12400] *= 3.0
        stats, gi, _ = run_full(prob, ix)
        hits = np.sum((gi[0] >= 12000) & (gi[0] < 12400))
        assert hits > 300, hits  # the winners really are concentrated


# ---- one-query CTAs: running cut bin, candidate bitmap, bin-ranked finish and slot merge

@pytest.mark.parametrize("S", [1, 100, 511, 512, 513, 700, 896])
def test_single_query_unsplit(S, bf16_ix, fp8_ix):
    # Up to 7 key tiles: one CTA, no split; the CTA ranks its candidates by bin itself and pads
    # rows that see fewer than 512 keys.
    for dtype, ix in ((inputs.BF16, bf16_ix), (inputs.FP8_E4M3, fp8_ix)):
        prob = inputs.make("q1", T=1, S=S, pos_offset=S - 1, seed=40 + S, dtype=dtype)
        stats, gi, gs = run_full(prob, ix)
        n = min(S, 512)
        assert np.all(gi[0, n:] == -1)
        if S <= 512:
            assert sorted(gi[0, :n].tolist()) == list(range(n))


@pytest.mark.parametrize("S", [5000, 30000])
def test_single_query_tie_storm(S, bf16_ix):
    # Every score is exactly 0 (one bin): the splits publish every tied key (S = 5000) or fall
    # back to an exact select (S = 30000), and the merge falls back to the radix path.
    prob = inputs.make("ties1", T=1, S=S, pos_offset=S - 1, seed=50, dtype=inputs.BF16)
    prob.k.zero_()
    stats, gi, gs = run_full(prob, bf16_ix)
    assert gi[0].tolist() == list(range(512))
    assert np.all(gs[0] == 0.0)


def test_single_query_all_negative(bf16_ix):
    prob = inputs.make("neg1", T=1, S=20000, pos_offset=19999, seed=51, dtype=inputs.BF16)
    prob.w.copy_(-prob.w.abs())
    stats, _, gs = run_full(prob, bf16_ix)
    assert np.all(gs[0] <= 0.0)


def test_single_query_wide_dynamic_range(fp8_ix):
    # A few keys scaled by 1e3 and 1e6 put the top bins hundreds of bins above the cut: the
    # published count windows are clipped to their top 256 bins (an undercount the merge allows).
    prob = inputs.make("wide1", T=1, S=30000, pos_offset=29999, seed=52, dtype=inputs.FP8_E4M3)
    g = torch.Generator().manual_seed(52)
    pick = torch.randperm(30000, generator=g)[:100]
    prob.kscale[pick[:50]] *= 1e6
    prob.kscale[pick[50:]] *= 1e3
    run_full(prob, fp8_ix)


def test_single_query_batched_splits_deterministic(fp8_ix):
    probs = [inputs.make(f"d{b}", T=1, S=40000, pos_offset=39999 - 977 * b, seed=60 + b,
                         dtype=inputs.FP8_E4M3) for b in range(8)]
    q = torch.stack([p.q for p in probs]).cuda()
    w = torch.stack([p.w for p in probs]).cuda()
    k = torch.stack([p.k for p in probs]).cuda()
    ks = torch.stack([p.kscale for p in probs]).cuda()
    pos = [p.pos_offset for p in probs]
    idx, sc = fp8_ix.score_topk_batched(q, w, k, ks, pos)
    fp8_ix.sync_status()
    for _ in range(3):
        idx2, sc2 = fp8_ix.score_topk_batched(q, w, k, ks, pos)
        fp8_ix.sync_status()
        assert torch.equal(idx, idx2) and torch.equal(sc, sc2)
    for b, prob in enumerate(probs):
        parity.check_rows(prob, [0], idx[b].cpu().numpy(), sc[b].cpu().numpy())


def test_single_query_clipped_windows(fp8_ix):
    # 2^50-fold key scales put a split's top bin ~400 bins above its cut: its count window is
    # clipped to the top 256 bins, its other candidates sit below the window, and the merge's
    # global cut falls below it, so the merge takes that split's whole list.
    prob = inputs.make("clip1", T=1, S=30000, pos_offset=29999, seed=53, dtype=inputs.FP8_E4M3)
    g = torch.Generator().manual_seed(53)
    pick = torch.randperm(30000, generator=g)[:40]
    prob.kscale[pick] *= 2.0 ** 50
    stats, gi, _ = run_full(prob, fp8_ix)
    # the scaled keys with a positive score (about half) lead the row
    assert len(set(pick.tolist()) & set(gi[0, :40].tolist())) >= 10


# ---- cases where the relative tolerance bites: scores far above 1

W_GAIN = 2.0 ** 12  # exact in fp32; I is positively homogeneous in w, so |I| grows to ~40


@pytest.mark.parametrize("dtype", [inputs.FP8_E4M3, inputs.BF16])
@pytest.mark.parametrize("T,S,pos", [(1001, 1001, 0), (300, 2000, 1700), (7, 5000, 2000),
                                     (1, 9000, 8999)])
def test_large_scores_relative_tolerance(dtype, T, S, pos, bf16_ix, fp8_ix):
    # With w scaled by 2^12 the scores reach tens, so eps * (1 + |I|) is a relative bound
    # (2% for FP8, 1e-4 for bf16) and the strict 1e-4 set rule is a relative check of the cut.
    # T > 1 runs the four-query kernel (ragged key tiles and query blocks, pos_offset > 0, a
    # split plan for T = 7); T = 1 the one-query kernel with its split merge.
    prob = inputs.make("big", T=T, S=S, pos_offset=pos, seed=70 + T, dtype=dtype)
    prob.w.mul_(W_GAIN)
    stats, _, gs = run_full(prob, _ix(prob, bf16_ix, fp8_ix))
    assert np.abs(gs[np.isfinite(gs)]).max() > 10.0  # the scale really is large
    assert stats["strict_set_diff"] == 0
    # fp32 accumulation of exactly decoded operands: far inside both tolerances (measured on
    # GB300: below 6e-6 for FP8, 1.6e-5 for bf16, whose tensor-core sums carry more terms)
    assert stats["max_rel_err"] < 5e-5, stats
    print(dtype, T, S, pos, stats)


# ---- bounded device waits: a lost arrival becomes DEVICE_TIMEOUT, not a hang

def test_device_timeout_is_reported_and_the_next_call_is_exact():
    # T = S = 4096: 1024 query blocks, no key split; the first CTA (the last queries) runs 32 key
    # tiles, so its score ring (28 tiles) wraps and the epilogue waits for the withheld release.
    prob = inputs.make("timeout", T=4096, S=4096, pos_offset=0, seed=80, dtype=inputs.BF16)
    with ds4idx.Indexer(ds4idx.BF16, max_T=4096, max_S=4096) as ix:
        dev = parity.to_device(prob)
        ix.debug_wait_test(1_000_000, withhold=True)  # 1 ms limit
        ix.score_topk(*dev, pos_offset=0)
        with pytest.raises(ds4idx.Ds4IdxError) as e:
            ix.sync_status()
        assert e.value.status == ds4idx.ERR_DEVICE_TIMEOUT
        ix.debug_wait_test(2_000_000_000, withhold=False)
        idx, sc = ix.score_topk(*dev, pos_offset=0)
        ix.sync_status()  # the error word was cleared: the normal call reports OK
        rows = inputs.sample_rows(prob.T, 80, n_random=128)
        stats = parity.check_rows(prob, rows, idx[rows].cpu().numpy(), sc[rows].cpu().numpy())
        assert stats["rows"] == len(rows)
