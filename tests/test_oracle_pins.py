"""Pins for the fp64 oracle: things other than the oracle itself that fix what it must return.

* a hand-computed worked example (tests/golden/hand_4x4.json),
* exact-rational brute force with rank-count selection (oracle/brute.py) on tiny inputs,
* decoders against closed forms and torch's own dtype casts,
* the special case H = 1, w = 1, which reduces to a numpy matmul + maximum + lexsort,
* invariants: causal masking, all-visible-kept, head permutation, positive scaling,
  FP8 scale placement, and the tie storm (all scores equal -> lowest indices).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import brute
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_4x4.json")


def bf16_codes(vals):
    return (torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
            .view(torch.int16).numpy().view(np.uint16))


def e4m3_codes(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _f(x):
    return -math.inf if x == "-inf" else float(x)


@pytest.fixture(scope="module")
def hand():
    with open(GOLDEN) as f:
        return json.load(f)


def _hand_inputs(g, dtype):
    enc = bf16_codes if dtype == orc.BF16 else e4m3_codes
    q = enc(g["q"])
    k = enc(g["k"])
    w = np.array(g["w"], dtype=np.float32)
    ks = np.array(g["fp8"]["kscale"], dtype=np.float32) if dtype == orc.FP8_E4M3 else None
    return q, w, k, ks


@pytest.mark.parametrize("dtype", [orc.BF16, orc.FP8_E4M3])
def test_hand_example_scores_and_topk(hand, dtype):
    q, w, k, ks = _hand_inputs(hand, dtype)
    gold = hand if dtype == orc.BF16 else hand["fp8"]
    sc = orc.scores(dtype, q, w, k, ks, pos_offset=0)
    for t, row in enumerate(gold["scores"]):
        assert sc[t, :len(row)].tolist() == row
        assert np.all(np.isneginf(sc[t, len(row):]))
    idx, val = orc.topk(dtype, q, w, k, ks, pos_offset=0, topk=2)
    assert idx.tolist() == gold["top2_idx"]
    assert val.tolist() == [[_f(x) for x in r] for r in gold["top2_score"]]
    if dtype == orc.BF16:
        idx1, _ = orc.topk(dtype, q, w, k, ks, pos_offset=0, topk=1)
        # Row t2 ties at 1.0 between keys 0 and 2: the lower index wins.
        assert idx1.tolist() == hand["top1_idx"]


@pytest.mark.parametrize("dtype", [orc.BF16, orc.FP8_E4M3])
def test_hand_example_brute(hand, dtype):
    q, w, k, ks = _hand_inputs(hand, dtype)
    gold = hand if dtype == orc.BF16 else hand["fp8"]
    ex = brute.exact_scores(dtype, q.tolist(), w.tolist(), k.tolist(),
                            None if ks is None else ks.tolist(), 0)
    for t, row in enumerate(gold["scores"]):
        assert [float(ex[(t, s)]) for s in range(len(row))] == row
    sel = brute.rank_count_topk(ex, 4, 4, 0, 2)
    assert [[s for s, _ in r] + [-1] * (2 - len(r)) for r in sel] == gold["top2_idx"]


def test_e4m3_decoder_all_codes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    for c in range(256):
        o = orc.decode_e4m3(c)
        r = float(ref[c])
        if c in (0x7F, 0xFF):
            assert math.isnan(o) and math.isnan(r)
            with pytest.raises(ValueError):
                brute.e4m3_value(c)
            continue
        assert o == r, hex(c)
        assert float(brute.e4m3_value(c)) == o
    # Closed forms of the OCP E4M3FN format.
    assert orc.decode_e4m3(0x7E) == 448.0
    assert orc.decode_e4m3(0xFE) == -448.0
    assert orc.decode_e4m3(0x01) == 2.0 ** -9
    assert orc.decode_e4m3(0x08) == 2.0 ** -6
    assert orc.decode_e4m3(0x38) == 1.0
    assert orc.decode_e4m3(0x80) == 0.0 and math.copysign(1, orc.decode_e4m3(0x80)) < 0


def test_bf16_decoder():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite only
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([orc.decode_bf16(int(b)) for b in bits])
    assert np.array_equal(got, ref.astype(np.float64))
    assert orc.decode_bf16(0x3F80) == 1.0 and orc.decode_bf16(0xC000) == -2.0


def _tiny(rng, dtype, T, S, H, D, integer):
    if integer:
        qv = rng.integers(-2, 3, size=(T, H, D)).astype(np.float32)
        kv = rng.integers(-2, 3, size=(S, D)).astype(np.float32)
        w = rng.choice([-1.0, -0.5, 0.5, 1.0, 2.0], size=(T, H)).astype(np.float32)
        ks = rng.choice([0.0, 0.25, 1.0, 2.0], size=S).astype(np.float32)
    else:
        qv = rng.standard_normal((T, H, D)).astype(np.float32)
        kv = rng.standard_normal((S, D)).astype(np.float32)
        w = rng.standard_normal((T, H)).astype(np.float32)
        ks = rng.uniform(0.0, 2.0, size=S).astype(np.float32)
    enc = bf16_codes if dtype == orc.BF16 else e4m3_codes
    return enc(qv), w, enc(kv), (ks if dtype == orc.FP8_E4M3 else None)


@pytest.mark.parametrize("dtype", [orc.BF16, orc.FP8_E4M3])
@pytest.mark.parametrize("seed", range(6))
def test_oracle_matches_exact_brute_force(dtype, seed):
    rng = np.random.default_rng(100 + seed)
    integer = seed % 2 == 1  # odd seeds: small integers, many exact ties
    T, S = int(rng.integers(3, 10)), int(rng.integers(4, 12))
    H, D = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    pos = int(rng.integers(0, 4))
    topk = int(rng.integers(1, 6))
    q, w, k, ks = _tiny(rng, dtype, T, S, H, D, integer)
    ex = brute.exact_scores(dtype, q.tolist(), w.tolist(), k.tolist(),
                            None if ks is None else ks.tolist(), pos)
    sc = orc.scores(dtype, q, w, k, ks, pos_offset=pos)
    for (t, s), v in ex.items():
        assert abs(sc[t, s] - float(v)) <= 1e-12 * (1 + abs(float(v))), (t, s)
    for t in range(T):
        n = min(pos + t, S - 1) + 1
        assert np.all(np.isneginf(sc[t, n:]))
    idx, val = orc.topk(dtype, q, w, k, ks, pos_offset=pos, topk=topk)
    sel = brute.rank_count_topk(ex, T, S, pos, topk)
    for t in range(T):
        want = [s for s, _ in sel[t]]
        assert idx[t, :len(want)].tolist() == want
        assert np.all(idx[t, len(want):] == -1)
        assert np.all(np.isneginf(val[t, len(want):]))


@pytest.mark.parametrize("seed", range(4))
def test_select_step_matches_rank_count(seed):
    rng = np.random.default_rng(seed)
    rows = rng.integers(-3, 4, size=(5, 23)).astype(np.float32)  # many ties
    rows[0] = 0.0
    rows[1, ::2] = -0.0  # signed zeros compare equal
    n_vis = np.array([23, 23, 17, 1, 9])
    for topk in (1, 5, 30):
        idx, _ = orc.select(rows, n_vis, topk)
        for r in range(rows.shape[0]):
            from fractions import Fraction
            ex = {(0, s): Fraction(float(rows[r, s])) for s in range(n_vis[r])}
            sel = brute.rank_count_topk(ex, 1, int(n_vis[r]), int(n_vis[r]) - 1, topk)[0]
            want = [s for s, _ in sel]
            assert idx[r, :len(want)].tolist() == want
            assert np.all(idx[r, len(want):] == -1)


def _random_problem(seed, T=40, S=40, H=8, D=16, dtype=orc.BF16):
    rng = np.random.default_rng(seed)
    return _tiny(rng, dtype, T, S, H, D, integer=False)


def test_single_head_reduces_to_matmul_relu_sort():
    rng = np.random.default_rng(7)
    T, S, D, pos = 30, 50, 16, 5
    qv = rng.standard_normal((T, 1, D)).astype(np.float32)
    kv = rng.standard_normal((S, D)).astype(np.float32)
    q, k = bf16_codes(qv), bf16_codes(kv)
    qd = torch.from_numpy(q.view(np.int16).copy()).view(torch.bfloat16).double().numpy()[:, 0]
    kd = torch.from_numpy(k.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    w = np.ones((T, 1), dtype=np.float32)
    ref = np.maximum(qd @ kd.T, 0.0)
    sc = orc.scores(orc.BF16, q, w, k, None, pos_offset=pos)
    idx, _ = orc.topk(orc.BF16, q, w, k, None, pos_offset=pos, topk=8)
    for t in range(T):
        n = min(pos + t, S - 1) + 1
        np.testing.assert_allclose(sc[t, :n], ref[t, :n], rtol=1e-12, atol=1e-14)
        order = np.lexsort((np.arange(n), -ref[t, :n]))[:8]
        # Zero scores tie; the lexsort tie-break on index matches the oracle's rule.
        assert idx[t, :min(8, n)].tolist() == order[:min(8, n)].tolist()


def test_causal_mask_invariance():
    q, w, k, _ = _random_problem(1)
    pos = 3
    base = orc.scores(orc.BF16, q, w, k, None, pos_offset=pos)
    bidx, _ = orc.topk(orc.BF16, q, w, k, None, pos_offset=pos, topk=6)
    for t in (0, 7, 20):
        p = pos + t
        k2 = k.copy()
        k2[p + 1:] = bf16_codes(np.full((k.shape[0] - p - 1, k.shape[1]), 3.0))
        sc2 = orc.scores(orc.BF16, q, w, k2, None, pos_offset=pos)
        assert np.array_equal(sc2[t], base[t])
        idx2, _ = orc.topk(orc.BF16, q, w, k2, None, pos_offset=pos, topk=6)
        assert np.array_equal(idx2[t], bidx[t])


def test_all_visible_kept_when_fewer_than_topk():
    q, w, k, _ = _random_problem(2)
    idx, val = orc.topk(orc.BF16, q, w, k, None, pos_offset=0, topk=64)
    for t in range(q.shape[0]):
        n = t + 1
        assert sorted(idx[t, :n].tolist()) == list(range(n))
        assert np.all(idx[t, n:] == -1) and np.all(np.isneginf(val[t, n:]))
        assert np.all(np.diff(val[t, :n]) <= 0)


def test_head_permutation_invariance():
    q, w, k, _ = _random_problem(3)
    perm = np.random.default_rng(0).permutation(q.shape[1])
    a = orc.scores(orc.BF16, q, w, k, None, pos_offset=2)
    b = orc.scores(orc.BF16, q[:, perm], w[:, perm], k, None, pos_offset=2)
    fin = np.isfinite(a)
    assert np.array_equal(fin, np.isfinite(b))
    np.testing.assert_allclose(b[fin], a[fin], rtol=1e-12, atol=1e-15)


def test_positive_weight_scaling():
    q, w, k, _ = _random_problem(4)
    a = orc.scores(orc.BF16, q, w, k, None, pos_offset=0)
    ia, _ = orc.topk(orc.BF16, q, w, k, None, pos_offset=0, topk=5)
    # Powers of two scale the fp32 weights exactly; 3.0 rounds each weight once (half an fp32
    # ulp per term), so there the bound is absolute, relative to the row's magnitude.
    fin = np.isfinite(a)
    for c, atol in ((2.0, 1e-15), (0.25, 1e-15), (3.0, 1e-6 * np.abs(a[fin]).max())):
        b = orc.scores(orc.BF16, q, (w * np.float32(c)).astype(np.float32), k, None)
        np.testing.assert_allclose(b[fin], c * a[fin], rtol=1e-12, atol=atol)
        ib, _ = orc.topk(orc.BF16, q, (w * np.float32(c)).astype(np.float32), k, None, topk=5)
        assert np.array_equal(ia, ib)


def test_fp8_scale_placement_and_bf16_agreement():
    # Values exact in both E4M3 and bf16: with kscale = 1 the two decoders must agree exactly,
    # and a power-of-two kscale[s] must scale column s exactly (scale after the head sum).
    rng = np.random.default_rng(5)
    T, S, H, D = 12, 20, 4, 8
    qv = rng.choice([-2.0, -1.0, -0.5, 0.0, 0.25, 1.0, 1.5], size=(T, H, D)).astype(np.float32)
    kv = rng.choice([-1.0, -0.5, 0.0, 0.5, 1.0, 2.0], size=(S, D)).astype(np.float32)
    w = rng.standard_normal((T, H)).astype(np.float32)
    one = np.ones(S, dtype=np.float32)
    a = orc.scores(orc.BF16, bf16_codes(qv), w, bf16_codes(kv), None)
    b = orc.scores(orc.FP8_E4M3, e4m3_codes(qv), w, e4m3_codes(kv), one)
    assert np.array_equal(a, b)
    ks = (2.0 ** rng.integers(-3, 4, size=S)).astype(np.float32)
    c = orc.scores(orc.FP8_E4M3, e4m3_codes(qv), w, e4m3_codes(kv), ks)
    fin = np.isfinite(a)
    assert np.array_equal(c[fin], (a * ks[None, :])[fin])


def test_tie_storm_picks_lowest_indices():
    q, w, _, _ = _random_problem(6, T=20, S=30)
    k = bf16_codes(np.zeros((30, 16)))
    idx, val = orc.topk(orc.BF16, q, w, k, None, pos_offset=10, topk=7)
    for t in range(20):
        n = min(10 + t, 29) + 1
        m = min(7, n)
        assert idx[t, :m].tolist() == list(range(m))
        assert np.all(val[t, :m] == 0.0)


def test_rejects_non_finite():
    q, w, k, _ = _random_problem(8, T=4, S=4)
    w = w.copy()
    w[1, 0] = np.nan
    with pytest.raises(ValueError):
        orc.scores(orc.BF16, q, w, k, None)
    q2, w2, k2, ks2 = _tiny(np.random.default_rng(0), orc.FP8_E4M3, 3, 3, 2, 2, False)
    ks2 = ks2.copy()
    ks2[0] = -1.0
    with pytest.raises(ValueError):
        orc.scores(orc.FP8_E4M3, q2, w2, k2, ks2)
