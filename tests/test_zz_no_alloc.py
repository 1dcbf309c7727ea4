"""The no-allocation entry point, checked against the handle-based one on the GPU.

ds4idx_score_topk_batched_noalloc serves callers that cannot allocate device memory when they
call the indexer, such as an engine that reserved all free HBM for its own pools or a framework
whose allocator must account for every byte. Its scratch is a fixed array inside the library.
The test calls it twice in a row through the C ABI, because the second call sees the array left
over from the first. Each time its outputs must equal those of ds4idx_score_topk_batched on the
same inputs: the same indices, and scores within the parity tolerance. The workloads use the
key-range split, which is what puts the scratch lists in play.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_lightning_indexer_gb300 import inputs
from sparse_attention_lightning_indexer_gb300 import ds4idx

from . import parity

pytestmark = pytest.mark.gpu


def _batch(dtype, T, S, positions, seed):
    probs = [inputs.make(f"na{b}", T=T, S=S, pos_offset=p, seed=seed + b, dtype=dtype)
             for b, p in enumerate(positions)]
    q = torch.stack([p.q for p in probs]).cuda()
    w = torch.stack([p.w for p in probs]).cuda()
    k = torch.stack([p.k for p in probs]).cuda()
    ks = torch.stack([p.kscale for p in probs]).cuda() if dtype == inputs.FP8_E4M3 else None
    return probs, q, w, k, ks


@pytest.mark.parametrize("dtype,T,S,positions", [
    (inputs.FP8_E4M3, 1, 9000, (8999, 4000, 700, 10)),   # batched decode, many splits
    (inputs.BF16, 6, 5000, (4994, 1200)),                # short chunks, split + merge
])
def test_noalloc_matches_handle_entry(dtype, T, S, positions):
    lib = ds4idx.load()
    probs, q, w, k, ks = _batch(dtype, T, S, positions, seed=40)
    B = len(probs)
    eps = parity.EPS[dtype]
    with ds4idx.Indexer(dtype, max_T=T, max_S=S, max_batch=B) as ix:
        ref_idx, ref_sc = ix.score_topk_batched(q, w, k, ks, positions)
        ix.sync_status()
    pos = (ctypes.c_int64 * B)(*positions)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        oi = torch.full((B, T, 512), -7, dtype=torch.int32, device="cuda")
        osc = torch.full((B, T, 512), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.ds4idx_score_topk_batched_noalloc(
            dtype, B, q.data_ptr(), w.data_ptr(), k.data_ptr(),
            None if ks is None else ks.data_ptr(), T, S, ctypes.cast(pos, ctypes.c_void_p), 512,
            oi.data_ptr(), osc.data_ptr(), stream)
        assert st == ds4idx.OK, (call, ds4idx.status_string(st))
        torch.cuda.synchronize()
        assert torch.equal(oi, ref_idx), f"call {call}: indices differ"
        got, want = osc.cpu().numpy(), ref_sc.cpu().numpy()
        fin = np.isfinite(want)
        assert np.array_equal(fin, np.isfinite(got)), f"call {call}: padding differs"
        assert np.all(np.abs(got[fin] - want[fin]) <= eps * (1 + np.abs(want[fin]))), call


def _noalloc_call(lib, dtype, q, w, k, ks, T, S, positions):
    B = len(positions)
    pos = (ctypes.c_int64 * B)(*positions)
    oi = torch.full((B, T, 512), -7, dtype=torch.int32, device="cuda")
    osc = torch.full((B, T, 512), float("nan"), dtype=torch.float32, device="cuda")
    st = lib.ds4idx_score_topk_batched_noalloc(
        dtype, B, q.data_ptr(), w.data_ptr(), k.data_ptr(),
        None if ks is None else ks.data_ptr(), T, S, ctypes.cast(pos, ctypes.c_void_p), 512,
        oi.data_ptr(), osc.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, oi, osc


def test_noalloc_matches_the_oracle():
    # One FP8 batched-decode case and one bf16 chunk case checked row by row against the fp64
    # oracle (score, set and order rules), not only against the handle entry point.
    lib = ds4idx.load()
    for dtype, T, S, positions in ((inputs.FP8_E4M3, 1, 7000, (6999, 2500, 300)),
                                   (inputs.BF16, 9, 3000, (2991, 40))):
        probs, q, w, k, ks = _batch(dtype, T, S, positions, seed=44)
        st, oi, osc = _noalloc_call(lib, dtype, q, w, k, ks, T, S, positions)
        assert st == ds4idx.OK, ds4idx.status_string(st)
        torch.cuda.synchronize()
        for b, prob in enumerate(probs):
            parity.check_rows(prob, list(range(T)), oi[b].cpu().numpy(), osc[b].cpu().numpy())


@pytest.mark.parametrize("T,pos", [(2048, 260096), (768, 262144 - 768)])
def test_noalloc_long_cache_chunks(T, pos):
    # Chunks on a 262144-key FP8 cache. The 2048-token chunk's split plan needs exactly the
    # array's 2^21 list words; the handle path would split the 768-token chunk into more lists
    # than the array holds, so here the split count steps down until they fit. Both must equal
    # the handle entry point's outputs.
    lib = ds4idx.load()
    S = 262144
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = ds4idx.plan_query(sms, 1, T, S, [pos], fixed_scratch=True)
    assert plan["list_words"] <= 1 << 21, plan
    probs, q, w, k, ks = _batch(inputs.FP8_E4M3, T, S, (pos,), seed=46)
    with ds4idx.Indexer(inputs.FP8_E4M3, max_T=T, max_S=S) as ix:
        ref_idx, ref_sc = ix.score_topk_batched(q, w, k, ks, [pos])
        ix.sync_status()
    for call in range(2):
        st, oi, osc = _noalloc_call(lib, inputs.FP8_E4M3, q, w, k, ks, T, S, (pos,))
        assert st == ds4idx.OK, (call, ds4idx.status_string(st))
        torch.cuda.synchronize()
        assert torch.equal(oi, ref_idx), f"call {call}: indices differ"
        assert torch.equal(osc, ref_sc), f"call {call}: scores differ"
    rows = [0, T // 2, T - 1]
    parity.check_rows(probs[0], rows, oi[0][rows].cpu().numpy(), osc[0][rows].cpu().numpy())


def test_noalloc_rejects_bad_arguments():
    lib = ds4idx.load()
    pos = (ctypes.c_int64 * 1)(0)
    p = ctypes.cast(pos, ctypes.c_void_p)
    s = torch.cuda.current_stream().cuda_stream
    # null inputs, bad dtype, bad topk: rejected before any work is enqueued
    assert lib.ds4idx_score_topk_batched_noalloc(0, 1, None, None, None, None, 4, 16, p, 512,
                                                 None, None, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_score_topk_batched_noalloc(5, 1, None, None, None, None, 4, 16, p, 512,
                                                 None, None, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_score_topk_batched_noalloc(0, 1, None, None, None, None, 4, 16, p, 128,
                                                 None, None, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_score_topk_batched_noalloc(0, 65, None, None, None, None, 4, 16, p, 512,
                                                 None, None, s) == ds4idx.ERR_INVALID_ARG
