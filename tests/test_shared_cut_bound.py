"""The lower bound behind the cut that one-query key splits share (Top-512 over a sequence whose
keys are split into n parts): if every part has at least k = ceil(512 / n) keys whose bin reaches
b_i, the lowest b_i is reached by at least n * k >= 512 keys of the sequence, so the sequence's
512th best key lies in that bin or above. The kernel raises each part's running cut to that bin
while the parts stream; the merge then needs exact counts only at and above the global cut bin,
which every part still has. These cases check the inequality on the bins the kernels use (the top
12 bits of the order-preserving map of an fp32 score), for random and adversarial key sets."""
import numpy as np
import pytest

TOPK = 512


def score_bins(scores: np.ndarray) -> np.ndarray:
    """12-bit bin of each fp32 score: the top bits of its order-preserving 32-bit code (-0 as +0)."""
    b = np.asarray(scores, dtype=np.float32).view(np.uint32).copy()
    b[b == 0x80000000] = 0
    neg = (b & 0x80000000) != 0
    o = np.where(neg, ~b, b | 0x80000000).astype(np.uint32)
    return (o >> 20).astype(np.int64)


def kth_best_bin(bins: np.ndarray, k: int) -> int:
    """The bin of a part's k-th best key (a part with fewer keys publishes nothing)."""
    return int(np.sort(bins)[::-1][k - 1])


def check(scores: np.ndarray, n_parts: int, bounds: list[int]):
    bins = score_bins(scores)
    k = -(-TOPK // n_parts)
    parts = np.split(bins, bounds) if bounds else np.array_split(bins, n_parts)
    assert len(parts) == n_parts
    published = [kth_best_bin(p, k) for p in parts if len(p) >= k]
    if len(published) < n_parts or len(bins) < TOPK:
        return  # some part never publishes: the cut is never raised
    low = min(published)
    global_cut = int(np.sort(bins)[::-1][TOPK - 1])
    assert low <= global_cut
    # at least 512 keys reach the shared bin (the argument's count)
    assert int((bins >= low).sum()) >= TOPK


@pytest.mark.parametrize("seed", range(20))
@pytest.mark.parametrize("n_parts", [2, 7, 19, 64])
def test_random_scores(seed, n_parts):
    rng = np.random.default_rng(seed)
    s = rng.normal(rng.normal(0, 0.004), 0.0064, size=n_parts * 700).astype(np.float32)
    check(s, n_parts, [])


@pytest.mark.parametrize("n_parts", [2, 19, 64])
def test_winners_in_one_part(n_parts):
    rng = np.random.default_rng(1)
    s = rng.normal(0, 1e-3, size=n_parts * 600).astype(np.float32)
    s[:TOPK] += 10.0  # every global winner in the first part
    check(s, n_parts, [])


@pytest.mark.parametrize("n_parts", [3, 19])
def test_ties_and_signs(n_parts):
    rng = np.random.default_rng(2)
    s = rng.choice(np.array([-1.0, -0.0, 0.0, 1e-30, 0.5, 0.5, 2.0], dtype=np.float32),
                   size=n_parts * 800)
    check(s, n_parts, [])


def test_uneven_parts():
    rng = np.random.default_rng(3)
    s = rng.standard_normal(20000).astype(np.float32)
    check(s, 5, [600, 5000, 5100, 19000])


def test_negative_scores_only():
    rng = np.random.default_rng(4)
    s = -np.abs(rng.standard_normal(19 * 800)).astype(np.float32)
    check(s, 19, [])


def test_bins_follow_score_order():
    s = np.array([-3.0, -1.0, -0.0, 0.0, 1e-38, 0.25, 1.0, 3.0], dtype=np.float32)
    b = score_bins(s)
    assert all(b[i] <= b[i + 1] for i in range(len(b) - 1))
    assert b[2] == b[3]  # -0 and +0 are the same score
