"""CPU model of the one-query (decode) selection: running cut bin, split slots, slot merge.

The CUDA kernel for one-query CTAs never orders words while it streams. It keeps a running cut
bin, publishes every key whose bin reaches its split's exact cut bin (grouped by bin, with a
window of per-bin counts), and the merging CTA finds a global cut bin G from the summed windows
and takes each list's prefix at or above G. This module restates those steps in numpy and
checks, on adversarial score distributions, that the result is exactly the 512 best words: the
argument the kernel's exactness rests on (a cut never passes the 512th best, undercounted
windows only lower G, a bin-grouped prefix is every word at or above G). Counter reads are made
stale on purpose, as concurrent warps see them. It tests the algorithm, not the CUDA code (the
GPU parity tests do that), and shares nothing with either implementation.
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


def highest_cut(counts, lo, hi):
    """Highest bin b in [lo, hi] with counts[b:hi+1].sum() >= K, else (lo, total)."""
    acc = 0
    for b in range(hi, lo - 1, -1):
        acc += int(counts[b])
        if acc >= K:
            return b, acc
    return lo, acc


def stream_split(words, rng, recut=64, stale_chunks=3):
    """Running cut over a split's words in 32-key chunks; counts read by the cut raise are a
    snapshot a few chunks old. Returns (candidate words, per-bin counts, cut, max bin)."""
    counts = np.zeros(4096, dtype=np.int64)
    cut, maxbin, own = 0, 0, 0
    snapshots = [counts.copy()]
    cands = []
    for c0 in range(0, len(words), 32):
        chunk = words[c0:c0 + 32]
        bn = bins(chunk)
        keep = bn >= cut
        if keep.any():
            kept = chunk[keep]
            cands.append(kept)
            np.add.at(counts, bn[keep], 1)
            maxbin = max(maxbin, int(bn[keep].max()))
            before, own = own, own + int(keep.sum())
            if own // recut != before // recut:
                snap = snapshots[max(0, len(snapshots) - 1 - int(rng.integers(0, stale_chunks + 1)))]
                view = np.minimum(snap, counts)          # a stale read never exceeds the truth
                b, cnt = highest_cut(view, cut, max(maxbin, cut))
                if cnt >= K and b > cut:
                    cut = b
        snapshots.append(counts.copy())
    cand = np.concatenate(cands) if cands else np.zeros(0, dtype=np.uint64)
    return cand, counts, cut, maxbin


def publish(words, rng):
    """One split's slot: (list grouped by bin from the top, window start, window counts)."""
    cand, counts, cut, maxbin = stream_split(words, rng)
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


def run_case(scores, n_splits, seed):
    rng = np.random.default_rng(seed)
    words = pack(scores, np.arange(len(scores)))
    parts = np.array_split(words, n_splits)
    got, path = merge([publish(p, rng) for p in parts])
    want = np.sort(words)[::-1][:K]
    assert np.array_equal(got, want)
    return path


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
