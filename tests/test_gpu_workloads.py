"""GPU parity at the full workload sizes, on sampled rows.

Each workload is run exactly as the benchmark launches it (one ds4idx call over the whole
workload), then a row sample (all t < 16, seeded random rows, the last 16) is checked against
the fp64 oracle with the score / set / order rules, and the selection is rerun on the kernel's
own fp32 scores for the same rows (tests/parity.py).
"""
import numpy as np
import pytest
import torch

from sparse_attention_lightning_indexer_gb300 import inputs
from sparse_attention_lightning_indexer_gb300 import ds4idx

from . import parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _check_workload(prob, n_random):
    ix = ds4idx.Indexer(prob.dtype, max_T=prob.T, max_S=prob.S)
    try:
        dev = parity.to_device(prob)
        idx, sc = ix.score_topk(*dev, pos_offset=prob.pos_offset)
        ix.sync_status()
        rows = inputs.sample_rows(prob.T, prob.meta["seed"], n_random=n_random)
        gi = idx[rows].cpu().numpy()
        gs = sc[rows].cpu().numpy()
        del idx, sc
        stats = parity.check_rows(prob, rows, gi, gs)
        dense = parity.dense_for_rows(ix, prob, dev, rows)
        parity.rerun_selection(prob, rows, dense, gi, gs)
        ix.sync_status()
    finally:
        ix.close()
        torch.cuda.empty_cache()
    return stats


def test_planted_16k():
    prob = inputs.workload("planted_16k")
    stats = _check_workload(prob, n_random=256)
    print("planted_16k", stats)


def test_prefill_64k_bench_configuration():
    prob = inputs.workload("prefill_64k")
    stats = _check_workload(prob, n_random=256)
    print("prefill_64k", stats)


def test_fp8_prefill_128k():
    prob = inputs.workload("fp8_prefill_128k")
    stats = _check_workload(prob, n_random=128)
    print("fp8_prefill_128k", stats, "strict FP8 set differences:", stats["strict_set_diff"])


def test_chunk_2048_at_260096():
    prob = inputs.workload("chunk_2048_at_260096")
    stats = _check_workload(prob, n_random=48)
    print("chunk_2048_at_260096", stats)


def test_decode_batch_8x262144():
    probs = inputs.decode_batch()
    B, S = len(probs), probs[0].S
    with ds4idx.Indexer(inputs.FP8_E4M3, max_T=1, max_S=S, max_batch=B) as ix:
        q = torch.stack([p.q for p in probs]).cuda()
        w = torch.stack([p.w for p in probs]).cuda()
        k = torch.stack([p.k for p in probs]).cuda()
        ks = torch.stack([p.kscale for p in probs]).cuda()
        idx, sc = ix.score_topk_batched(q, w, k, ks, [p.pos_offset for p in probs])
        ix.sync_status()
        for b, prob in enumerate(probs):
            gi, gs = idx[b].cpu().numpy(), sc[b].cpu().numpy()
            parity.check_rows(prob, [0], gi, gs)
            dense = ix.score_dense_debug(q[b], w[b], k[b], ks[b], prob.pos_offset)
            parity.rerun_selection(prob, [0], dense.cpu().numpy(), gi, gs)
        ix.sync_status()
