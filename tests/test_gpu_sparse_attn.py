"""GPU parity of sparse attention over the selected keys (ds4idx_sparse_attention, through the
C ABI) against the fp64 oracle (oracle.sparse_attention).

Tolerance, from the arithmetic: the kernel's scores are fp32 sums of exact bf16 products, its
probabilities are fp32 then rounded to bf16 (relative error <= 2^-9) before the value product,
and the output is rounded to bf16 (<= 2^-9 relative). So per output element
    |o_gpu - o| <= 2^-9 * sum_j p_j |v_j| + 2^-9 |o| + (fp32 terms),
checked with a factor 2 margin: 2^-8 * sum_j p_j |v_j| + 2^-8 |o| + 1e-6, where p_j comes from
the oracle's own lse. lse: |d lse| <= 1e-4 + 1e-5 |lse| (fp32 sums and the exponent's rounding).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_attention_lightning_indexer_gb300 import ds4idx

pytestmark = pytest.mark.gpu

H, DQK, DV, K = 128, 576, 512, 512


def _inputs(T, R, seed, n_valid=None, q_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, H, DQK, generator=g) * q_scale).to(torch.bfloat16)
    kv = torch.randn(R, DQK, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    idx = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        n = K if n_valid is None else n_valid[t % len(n_valid)]
        sel = rng.choice(R, size=min(n, R), replace=False)
        slots = rng.choice(K, size=sel.size, replace=False)
        idx[t, slots] = sel
    return q, kv, idx


def _check(q, kv, idx, scale, out, lse, row0=None):
    T = q.shape[0]
    o_ref, l_ref = orc.sparse_attention(q, kv, idx, scale, DV, row0=row0)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    qf, kf = q.double().numpy(), kv.double().numpy()
    for t in range(T):
        rows = idx[t][idx[t] >= 0].astype(np.int64) + (0 if row0 is None else int(row0[t]))
        if rows.size == 0:
            assert np.all(o[t] == 0) and np.all(np.isneginf(l[t])), t
            continue
        s = scale * qf[t] @ kf[rows].T                      # [H, n]
        p = np.exp(s - l_ref[t][:, None])
        a = p @ np.abs(kf[rows, :DV])                       # sum_j p_j |v_j|
        bound = 2.0 ** -8 * a + 2.0 ** -8 * np.abs(o_ref[t]) + 1e-6
        err = np.abs(o[t] - o_ref[t])
        bad = np.argwhere(err > bound)
        assert bad.size == 0, (t, bad[:3], err[tuple(bad[0])], bound[tuple(bad[0])])
        np.testing.assert_array_less(np.abs(l[t] - l_ref[t]), 1e-4 + 1e-5 * np.abs(l_ref[t]))


@pytest.mark.parametrize("T,R,n_valid,q_scale", [
    (3, 600, None, 1.0),            # full 512-key sets
    (37, 5000, [512, 3, 1, 0, 200, 511], 1.0),  # ragged sets, one empty row
    (16, 2000, None, 4.0),          # peaked softmax (large scores)
])
def test_sparse_attention_matches_oracle(T, R, n_valid, q_scale):
    q, kv, idx = _inputs(T, R, seed=T, n_valid=n_valid, q_scale=q_scale)
    scale = DQK ** -0.5
    out, lse = ds4idx.sparse_attention(q.cuda(), kv.cuda(), torch.from_numpy(idx).cuda(), scale)
    ds4idx.sparse_attention_status()
    _check(q, kv, idx, scale, out, lse)


def test_sparse_attention_row_offsets_and_bad_positions():
    # Two sequences in one pool (row0 per token); positions past the pool count as empty.
    T, R = 8, 3000
    q, kv, idx = _inputs(T, 1200, seed=5)
    row0 = np.array([0, 0, 0, 0, 1500, 1500, 1500, 1500], dtype=np.int64)
    kv_pool = torch.cat([kv, torch.zeros(300, DQK, dtype=torch.bfloat16), kv, kv[:300]])
    idx_bad = idx.copy()
    idx_bad[6, 7] = 5000  # row 6500 > pool: empty
    want_idx = idx_bad.copy()
    want_idx[6, 7] = -1
    out, lse = ds4idx.sparse_attention(q.cuda(), kv_pool.cuda(), torch.from_numpy(idx_bad).cuda(),
                                       0.05, kv_row0=torch.from_numpy(row0).cuda())
    ds4idx.sparse_attention_status()
    _check(q, kv_pool, want_idx, 0.05, out, lse, row0=row0)


def test_sparse_attention_rejects_bad_arguments():
    lib = ds4idx.load()
    q = torch.zeros((1, H, DQK), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((10, DQK), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((1, K), dtype=torch.int32, device="cuda")
    out = torch.zeros((1, H, DV), dtype=torch.bfloat16, device="cuda")
    P = lambda t: t.data_ptr()  # noqa: E731
    s = torch.cuda.current_stream().cuda_stream
    assert lib.ds4idx_sparse_attention(P(q), P(kv), 10, P(idx), None, 1, 64, DQK, DV, K, 1.0,
                                       P(out), None, s) == ds4idx.ERR_UNSUPPORTED
    assert lib.ds4idx_sparse_attention(None, P(kv), 10, P(idx), None, 1, H, DQK, DV, K, 1.0,
                                       P(out), None, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_sparse_attention(P(q), P(kv), 10, P(idx), None, 1, H, DQK, DV, K, 0.0,
                                       P(out), None, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_sparse_attention(P(q), P(kv), 10, P(idx), None, 0, H, DQK, DV, K, 1.0,
                                       P(out), None, s) == ds4idx.OK
