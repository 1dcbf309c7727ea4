"""Pins of the oracle's sparse attention (oracle.sparse_attention) against things other than
itself: hand-worked cases (tests/golden/sparse_attn_hand.json), dense attention over all keys
with the unselected ones masked to -inf (a different computation: no gather, a full score row,
numpy's float64 matmul and exp), closed forms (one key, equal scores), invariance under the
order of the index list, and homogeneity in the values.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sparse_attn_hand.json")


def test_hand_cases():
    with open(GOLDEN) as f:
        g = json.load(f)
    kv = torch.tensor(g["kv"], dtype=torch.bfloat16)
    for c in g["cases"]:
        q = torch.tensor([[c["q"]]], dtype=torch.bfloat16)
        idx = np.array([c["idx"]], dtype=np.int32)
        o, lse = orc.sparse_attention(q, kv, idx, c["scale"], 1)
        assert o[0, 0, 0] == pytest.approx(c["o"], abs=1e-15), c
        want = -np.inf if c["lse"] == "-inf" else c["lse"]
        assert lse[0, 0] == pytest.approx(want, abs=1e-15), c


def _rand(T, H, D, R, K, seed):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, H, D, generator=g) * 0.3).to(torch.bfloat16)
    kv = (torch.randn(R, D, generator=g) * 0.3).to(torch.bfloat16)
    idx = np.stack([np.random.default_rng(seed + t).choice(R, size=K, replace=False)
                    for t in range(T)]).astype(np.int32)
    idx[0, ::3] = -1
    return q, kv, idx


@pytest.mark.parametrize("seed", [0, 1])
def test_matches_masked_dense_attention(seed):
    T, H, D, Dv, R, K = 5, 4, 24, 16, 60, 17
    q, kv, idx = _rand(T, H, D, R, K, seed)
    scale = 0.37
    o, lse = orc.sparse_attention(q, kv, idx, scale, Dv)
    qf, kf = q.double().numpy(), kv.double().numpy()
    for t in range(T):
        sel = np.zeros(R, dtype=bool)
        sel[idx[t][idx[t] >= 0]] = True
        s = scale * qf[t] @ kf.T                     # [H, R]: every key scored
        s = np.where(sel[None, :], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / e.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(o[t], p @ kf[:, :Dv], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t], (m[:, 0] + np.log(e.sum(axis=1))), rtol=0, atol=1e-12)


def test_closed_forms():
    R, D, Dv = 30, 8, 6
    _, kv, _ = _rand(1, 1, D, R, 4, 3)
    kf = kv.double().numpy()
    # one selected key: its value, lse = its score
    q = (torch.randn(1, 2, D, generator=torch.Generator().manual_seed(1)) * 0.5).to(torch.bfloat16)
    o, lse = orc.sparse_attention(q, kv, np.array([[-1, 7, -1]], dtype=np.int32), 0.5, Dv)
    np.testing.assert_array_equal(o[0, 0], kf[7, :Dv])
    assert lse[0, 1] == pytest.approx(0.5 * float(q[0, 1].double() @ kv[7].double()), abs=1e-14)
    # equal scores (q = 0): the mean of the selected values
    sel = [3, 9, 11, 2]
    o, lse = orc.sparse_attention(torch.zeros(1, 1, D, dtype=torch.bfloat16), kv,
                                  np.array([sel], dtype=np.int32), 1.0, Dv)
    np.testing.assert_allclose(o[0, 0], kf[sel, :Dv].mean(axis=0), atol=1e-15)
    assert lse[0, 0] == pytest.approx(np.log(4), abs=1e-15)


def test_order_and_row_offset_invariance():
    T, H, D, Dv, R, K = 3, 2, 16, 8, 40, 9
    q, kv, idx = _rand(T, H, D, R, K, 5)
    o1, l1 = orc.sparse_attention(q, kv, idx, 0.3, Dv)
    perm = idx[:, ::-1].copy()
    o2, l2 = orc.sparse_attention(q, kv, perm, 0.3, Dv)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)
    # the same keys placed 10 rows further into a bigger pool, with row0 = 10
    kv2 = torch.cat([torch.zeros(10, D, dtype=torch.bfloat16), kv])
    o3, l3 = orc.sparse_attention(q, kv2, idx, 0.3, Dv, row0=np.full(T, 10))
    np.testing.assert_array_equal(o1, o3)
    np.testing.assert_array_equal(l1, l3)


def test_rejects_rows_outside_the_pool():
    q, kv, idx = _rand(1, 1, 8, 10, 3, 0)
    idx[0, 0] = 10
    with pytest.raises(ValueError):
        orc.sparse_attention(q, kv, idx, 1.0, 4)
