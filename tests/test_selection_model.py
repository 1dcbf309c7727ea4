"""CPU model of the one-query (decode) selection: running cut bin, split slots, slot merge.

The CUDA kernel for one-query CTAs never orders words while it streams. It keeps a running cut
bin, publishes every key whose bin reaches its split's exact cut bin (grouped by bin, with a
window of per-bin counts), and the merging CTA finds a global cut bin G from the summed windows
and takes each list's prefix at or above G. This module restates those steps in numpy and
checks, on adversarial score distributions, that the result is exactly the 512 best words: the
argument the kernel's exactness rests on (a cut never passes the 512th best, undercounted
windows only lower G, a bin-grouped prefix is every word at or above G). Counter reads are made
stale on purpose, as concurrent warps see them. The splits of a sequence may also share their cut:
they stream side by side, each publishes the bin its ceil(512 / splits)-th best counted key
reaches, and once all have published each raises its cut to the lowest of those bins; those
cases check that the merge stays exact when a split's cut passes its own 512th best. It tests the
algorithm, not the CUDA code (the GPU parity tests do that), and shares nothing with either
implementation.
"""
import numpy as np
import pytest

K = 512
SLOT_CAP = 1022      # published words per split at most
WINDOW = 256         # bins in a split's count window
SURV_CAP = 2048      # words the merge ranks directly
RANK_BINS = 2048     # bins the merge's ranking spans at most


def pack(scores, idx):
    """(score, index) -> order-preserving u64 words (score code << 32 | ~index)."""
    b = np.asarray(scores, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = np.where(b == 0x80000000, 0, b)
    code = np.where(b & 0x80000000, (~b) & 0xFFFFFFFF, b | 0x80000000)
    return (code << np.uint64(32)) | ((~np.asarray(idx, dtype=np.uint64)) & np.uint64(0xFFFFFFFF))


def bins(words):
    return (np.asarray(words, dtype=np.uint64) >> np.uint64(52)).astype(np.int64)


def highest_cut(counts, lo, hi, k=K):
    """Highest bin b in [lo, hi] with counts[b:hi+1].sum() >= k, else (lo, total)."""
    run = np.cumsum(counts[lo:hi + 1][::-1])
    hit = np.flatnonzero(run >= k)
    if hit.size:
        return hi - int(hit[0]), int(run[hit[0]])
    return lo, int(run[-1]) if run.size else 0


class SplitStream:
    """A split's running cut over its words in 32-key chunks; counts read by a cut raise are a
    snapshot a few chunks old (a stale read never exceeds the truth)."""

    def __init__(self, words, rng, recut=64, stale_chunks=3):
        self.words, self.rng, self.recut, self.stale = words, rng, recut, stale_chunks
        self.counts = np.zeros(4096, dtype=np.int64)
        self.cut, self.maxbin, self.own, self.pos = 0, 0, 0, 0
        self.snapshots = [self.counts.copy()]
        self.cands = []

    def done(self):
        return self.pos >= len(self.words)

    def stale_counts(self):
        back = int(self.rng.integers(0, self.stale + 1))
        return np.minimum(self.snapshots[max(0, len(self.snapshots) - 1 - back)], self.counts)

    def step(self):
        """One chunk: keys at or above the cut are listed and counted; every `recut` listed keys
        the cut is raised to the highest bin that 512 counted keys reach."""
        chunk = self.words[self.pos:self.pos + 32]
        self.pos += 32
        bn = bins(chunk)
        keep = bn >= self.cut
        if keep.any():
            self.cands.append(chunk[keep])
            np.add.at(self.counts, bn[keep], 1)
            self.maxbin = max(self.maxbin, int(bn[keep].max()))
            before, self.own = self.own, self.own + int(keep.sum())
            if self.own // self.recut != before // self.recut:
                b, cnt = highest_cut(self.stale_counts(), self.cut, max(self.maxbin, self.cut))
                if cnt >= K and b > self.cut:
                    self.cut = b
        self.snapshots.append(self.counts.copy())

    def result(self):
        cand = np.concatenate(self.cands) if self.cands else np.zeros(0, dtype=np.uint64)
        return cand, self.counts, self.cut, self.maxbin


def stream_split(words, rng):
    """One split streamed alone. Returns (candidate words, per-bin counts, cut, max bin)."""
    s = SplitStream(words, rng)
    while not s.done():
        s.step()
    return s.result()


def stream_shared(parts, rng, wake=0.5, stale_pub=4, rate=None):
    """The splits of one sequence streamed side by side at uneven rates, with the cut they share:
    while its keys stream, each split now and then publishes the bin that its k-th best counted
    key reaches (k = ceil(512 / splits), from a stale count read) and, once every split has
    published, raises its cut to the lowest published bin (read from a stale copy of the
    published bins, which only rise). `rate` gives the splits' relative speeds (default: random).
    Returns each split's stream result."""
    ns = len(parts)
    k = -(-K // ns)
    splits = [SplitStream(p, rng) for p in parts]
    pub = np.zeros(ns, dtype=np.int64)  # bin + 1, 0 = not yet published
    pub_history = [pub.copy()]
    rate = rng.uniform(0.5, 1.5, size=ns) if rate is None else np.asarray(rate, dtype=np.float64)
    while True:
        live = [i for i in range(ns) if not splits[i].done()]
        if not live:
            break
        w = rate[live] / rate[live].sum()
        i = live[int(rng.choice(len(live), p=w))]
        s = splits[i]
        s.step()
        if s.done() or rng.random() >= wake:
            continue  # the raise only runs while the split's keys stream
        b, cnt = highest_cut(s.stale_counts(), s.cut, max(s.maxbin, s.cut), k)
        if cnt >= k and b + 1 > pub[i]:
            pub[i] = b + 1
            pub_history.append(pub.copy())
        seen = pub_history[max(0, len(pub_history) - 1 - int(rng.integers(0, stale_pub + 1)))]
        low = int(seen.min())
        if low > 0 and low - 1 > s.cut:
            s.cut = low - 1
    return [s.result() for s in splits]


def publish(words, streamed, rng):
    """One split's slot from its stream: (list grouped by bin from the top, window start, window
    counts)."""
    cand, counts, cut, maxbin = streamed
    bstar, m = highest_cut(counts, cut, max(maxbin, cut))
    if m <= SLOT_CAP:
        out = cand[bins(cand) >= bstar]
        assert len(out) == m
        wlo = maxbin - (WINDOW - 1) if maxbin - bstar >= WINDOW else bstar
        win = counts[wlo:maxbin + 1].copy() if m else np.zeros(0, dtype=np.int64)
    else:  # fallback: the split's exact 512 best, window counted from them
        out = np.sort(words)[::-1][:K]
        hi = int(bins(out).max()) if len(out) else 0
        wlo = max(0, hi - (WINDOW - 1))
        win = np.bincount(bins(out)[bins(out) >= wlo] - wlo, minlength=hi - wlo + 1) if len(out) else np.zeros(0)
    # grouped by bin: window bins from the top, each bin's words in any (here random) order
    bn = bins(out)
    bucket = np.where(bn >= wlo, int(wlo + len(win) - 1) - bn, len(win))
    order = np.lexsort((rng.random(len(out)), bucket))
    return out[order], int(wlo), np.asarray(win, dtype=np.int64)


def merge(slots):
    lo_all = [lo for lst, lo, win in slots if len(win)]
    H = max((lo + len(win) - 1 for lst, lo, win in slots if len(win)), default=0)
    L = min(lo_all) if lo_all else 0
    mh = np.zeros(4096, dtype=np.int64)
    for lst, lo, win in slots:
        mh[lo:lo + len(win)] += win
    G, c = highest_cut(mh, min(L, H), H)
    if c < K:
        G = 0
    prefixes = []
    for lst, lo, win in slots:
        n = len(lst) if G <= lo else int(win[G - lo:].sum())
        prefixes.append(lst[:n])
    surv = np.concatenate(prefixes) if prefixes else np.zeros(0, dtype=np.uint64)
    sb = bins(surv)
    surv = surv[(sb >= G) & (sb <= H)]
    if len(surv) <= SURV_CAP and H - G < RANK_BINS:
        return np.sort(surv)[::-1][:K], "ranked"
    everything = np.concatenate([lst for lst, lo, win in slots])
    return np.sort(everything)[::-1][:K], "fallback"


def run_case(scores, n_splits, seed, shared=False, with_total=False, bounds=None, **shared_opts):
    """Stream, publish and merge; the merged words must be exactly the 512 best. With `shared`,
    the splits stream side by side and share their cut (`shared_opts` go to `stream_shared`).
    `bounds` splits the keys at the given positions instead of evenly. Returns the merge's path
    (and, with `with_total`, the number of words the splits published)."""
    rng = np.random.default_rng(seed)
    words = pack(scores, np.arange(len(scores)))
    parts = np.split(words, bounds) if bounds else np.array_split(words, n_splits)
    assert len(parts) == n_splits
    if shared:
        streams = stream_shared(parts, rng, **shared_opts)
    else:
        streams = [stream_split(p, rng) for p in parts]
    want = np.sort(words)[::-1][:K]
    if len(words) >= K:  # no split's cut passes the sequence's 512th best
        assert max(cut for _, _, cut, _ in streams) <= int(bins(want[-1:])[0])
    slots = [publish(p, s, rng) for p, s in zip(parts, streams)]
    got, path = merge(slots)
    assert np.array_equal(got, want)
    return (path, sum(len(lst) for lst, _, _ in slots)) if with_total else path


def _gauss(n, seed, mean=0.0):
    return (np.random.default_rng(seed).standard_normal(n) * 0.0078 + mean).astype(np.float32)


def test_pack_orders_like_the_selection_rule():
    s = np.array([1.0, -1.0, 0.0, -0.0, 1.0, 2.5e-3], dtype=np.float32)
    w = pack(s, np.arange(6))
    order = np.argsort(w)[::-1]
    # best first: 1.0 (idx 0 before idx 4), 2.5e-3, then +0 and -0 as equal scores (idx 2, 3)
    assert order.tolist() == [0, 4, 5, 2, 3, 1]
    assert np.all(np.diff(bins(np.sort(w))) >= 0)  # bins are monotone in the word


@pytest.mark.parametrize("seed", range(4))
def test_gaussian_scores_split_19(seed):
    assert run_case(_gauss(19 * 1400, seed), 19, seed) == "ranked"


def test_scores_skewed_negative():
    # most scores negative: the running cut must climb through the negative bins
    run_case(_gauss(19 * 1400, 7, mean=-0.02), 19, 7)


def test_all_negative_scores():
    run_case(-np.abs(_gauss(12000, 8)), 9, 8)


def test_tie_storm_takes_the_fallback():
    s = np.zeros(19 * 1400, dtype=np.float32)
    assert run_case(s, 19, 9) == "fallback"


def test_outliers_clip_the_windows():
    # a few keys far above the rest put some splits' top bins 80-160 bins over their cuts, and
    # the merge's G sits among the normal keys, far below those splits' top bins
    s = _gauss(19 * 1400, 10)
    rng = np.random.default_rng(10)
    pick = rng.choice(len(s), 100, replace=False)
    s[pick[:50]] *= np.float32(1e6)
    s[pick[50:]] *= np.float32(1e3)
    run_case(s, 19, 10)


def test_concentrated_winners_in_one_split():
    s = _gauss(19 * 1400, 11)
    s[3 * 1400:3 * 1400 + 450] += np.float32(0.05)
    run_case(s, 19, 11)


@pytest.mark.parametrize("n", [1, 300, 511, 512, 513, 2000])
def test_few_keys(n):
    run_case(_gauss(n, 12 + n), 1 if n < 1000 else 4, n)


def test_huge_outliers_clip_windows_below_the_cut():
    # 2^50-fold outliers put a split's top bin ~400 bins above its cut: its window is clipped,
    # its normal candidates sit below the window, and G (set by the normal winners) is below it
    s = _gauss(19 * 1400, 13)
    rng = np.random.default_rng(13)
    s[rng.choice(len(s), 40, replace=False)] *= np.float32(2.0 ** 50)
    run_case(s, 19, 13)


def test_winners_in_one_split_at_its_cut():
    # every global winner comes from split 0, whose scores crowd a few bins: the split's cut bin
    # holds part of the global Top-512, including keys that arrive after the cut reached it
    s = _gauss(19 * 1400, 14) * np.float32(0.01)
    s[:1400] = np.float32(1.0) + np.random.default_rng(14).random(1400).astype(np.float32) * np.float32(0.3)
    run_case(s, 19, 14)


@pytest.mark.parametrize("seed", range(3))
def test_single_split(seed):
    run_case(_gauss(13824, 20 + seed), 1, seed)


# ---- the cut shared by the splits of a sequence

def _own_cut_bins(parts):
    """Each split's own 512th-best bin: as high as its cut can rise without the shared cut."""
    return [int(bins(np.sort(p)[::-1][K - 1:K])[0]) if len(p) >= K else 0 for p in parts]


@pytest.mark.parametrize("seed", range(4))
def test_shared_cut_lists_fewer_words(seed):
    s = _gauss(19 * 1400, seed)
    path, shared = run_case(s, 19, seed, shared=True, with_total=True)
    _, alone = run_case(s, 19, seed, with_total=True)
    assert path == "ranked" and shared < alone
    # the shared cut takes splits' cuts past their own 512th best
    parts = np.array_split(pack(s, np.arange(len(s))), 19)
    cuts = [r[2] for r in stream_shared(parts, np.random.default_rng(seed))]
    assert any(c > own for c, own in zip(cuts, _own_cut_bins(parts)))


@pytest.mark.parametrize("case", ["skewed", "negative", "outliers", "huge_outliers",
                                  "concentrated", "one_split_at_its_cut"])
def test_shared_cut_adversarial(case):
    rng = np.random.default_rng(40)
    s = _gauss(19 * 1400, 40)
    if case == "skewed":
        s = _gauss(19 * 1400, 41, mean=-0.02)
    elif case == "negative":
        s = -np.abs(s)
    elif case == "outliers":
        pick = rng.choice(len(s), 100, replace=False)
        s[pick[:50]] *= np.float32(1e6)
        s[pick[50:]] *= np.float32(1e3)
    elif case == "huge_outliers":
        s[rng.choice(len(s), 40, replace=False)] *= np.float32(2.0 ** 50)
    elif case == "concentrated":
        s[3 * 1400:3 * 1400 + 450] += np.float32(0.05)
    else:
        s *= np.float32(0.01)
        s[:1400] = np.float32(1.0) + rng.random(1400).astype(np.float32) * np.float32(0.3)
    run_case(s, 19, 40, shared=True)


def test_shared_cut_tie_storm_takes_the_fallback():
    assert run_case(np.zeros(19 * 1400, dtype=np.float32), 19, 42, shared=True) == "fallback"


def test_shared_cut_winners_last_in_the_slowest_split():
    # every global winner sits at the end of split 0, which streams at a third of the others'
    # rate: the others publish and raise their cuts from noise long before the winners arrive
    s = _gauss(19 * 1400, 43)
    s[1400 - 450:1400] += np.float32(0.05)
    rate = np.full(19, 1.5)
    rate[0] = 0.5
    run_case(s, 19, 43, shared=True, rate=rate)


def test_shared_cut_split_too_small_to_publish():
    # the last split holds fewer than ceil(512 / 19) = 27 keys: it never publishes, so no split's
    # cut passes its own 512th best, and the merge is still exact
    s = _gauss(18 * 1400 + 20, 44)
    bounds = [1400 * i for i in range(1, 19)]
    parts = np.split(pack(s, np.arange(len(s))), bounds)
    cuts = [r[2] for r in stream_shared(parts, np.random.default_rng(44))]
    assert all(c <= own for c, own in zip(cuts, _own_cut_bins(parts)))
    assert run_case(s, 19, 44, shared=True, bounds=bounds) == "ranked"


@pytest.mark.parametrize("seed", range(3))
def test_shared_cut_eager_publishing_stale_reads(seed):
    run_case(_gauss(19 * 1400, 45 + seed), 19, seed, shared=True, wake=1.0, stale_pub=16)


@pytest.mark.parametrize("n_splits", [2, 64])
def test_shared_cut_split_counts(n_splits):
    run_case(_gauss(n_splits * 900, 48 + n_splits), n_splits, n_splits, shared=True)


def test_shared_cut_decode_sized_split():
    # 19 splits of 13,824 keys, as one sequence of 262,144 keys is split on 152 SMs
    path, shared = run_case(_gauss(19 * 13824, 50), 19, 50, shared=True, with_total=True)
    assert path == "ranked" and shared < 4000
