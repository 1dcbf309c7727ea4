"""The synthetic workloads do what they are for, checked with the oracle alone (no GPU).

The 16k workload plants 32 topic keys per aligned 1024-key block and lifts one query in eight
towards a topic, so that its Top-512 is not a random sample of the row: the oracle's own Top-512
of the planted queries must hold most of their visible same-topic keys.
"""
import numpy as np

from oracle import oracle as orc
from sparse_attention_lightning_indexer_gb300 import inputs

from . import parity


def test_planted_keys_reach_the_oracle_top512():
    prob = inputs.workload("planted_16k")
    q_rows = np.sort(prob.meta["planted_queries"].numpy())
    rows = q_rows[::32]  # 64 planted queries spread over the sequence
    q, k = prob.codes()
    idx, _ = orc.topk(prob.dtype, q, prob.w.numpy(), k, None, prob.pos_offset, prob.topk, rows)
    rate, n = parity.planted_hit_rate(prob, {int(t): idx[r] for r, t in enumerate(rows)})
    assert n > 500
    assert rate > 0.75, rate
    # Unplanted queries of the same rows' neighbourhood do not favour the planted keys: their
    # share of planted keys in the Top-512 stays near the planted density (32 / 1024).
    others = np.setdiff1d(np.arange(8192, 16384, 512), q_rows)[:16]
    idx_o, _ = orc.topk(prob.dtype, q, prob.w.numpy(), k, None, prob.pos_offset, prob.topk,
                        others)
    planted = set(prob.meta["planted_keys"].tolist())
    share = np.mean([np.isin(r, list(planted)).mean() for r in idx_o])
    assert share < 0.1, share
