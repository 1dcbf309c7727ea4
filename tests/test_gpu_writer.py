"""GPU parity of the FP8 index-cache writer (ds4idx_quantize_keys / ds4idx_quantize_queries,
through the C ABI) against the oracle: codes, scales and folded weights must be bit-exact.

Cases: ragged row counts, fp32 and bf16 inputs, rows that are all zero, rows with negative
zeros, exact ties between E4M3 codes, values that saturate, scattered slot mappings with padding
(-1) and out-of-range slots, in-place weight folding, and the FP8 workloads' own shapes, whose
writer output must also equal the workload codes the benchmark and the indexer tests use.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_attention_lightning_indexer_gb300 import ds4idx, inputs

pytestmark = pytest.mark.gpu


def _special_rows(n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 128, generator=g) * torch.exp(torch.randn(n, 1, generator=g) * 3)
    x[0] = 0.0                                   # scale 0 -> codes 0
    x[1, ::2] = -0.0                             # negative zeros in a non-zero row
    x[2] = torch.arange(128, dtype=torch.float32) - 64.0   # integers: exact ties after scaling
    x[3, 0] = 1e30                               # one huge value, the rest flush to zero
    x[4] = 1e-30                                 # tiny but non-zero (subnormal scale range)
    x[5, :] = 448.0
    x[5, 1] = -448.0
    return x


def _oracle_keys(x):
    xf = x.float().numpy()
    return orc.quantize_rows(xf)


@pytest.mark.parametrize("in_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", [1, 7, 10007])
def test_keys_contiguous(in_dtype, n):
    x = _special_rows(max(n, 6), 1)[:n].to(in_dtype)
    R = n + 100
    kc = torch.full((R, 128), 0xAB, dtype=torch.uint8, device="cuda")
    ks = torch.full((R,), -1.0, dtype=torch.float32, device="cuda")
    ds4idx.quantize_keys(x.cuda(), kc, ks, dst_offset=50)
    torch.cuda.synchronize()
    codes, scales = _oracle_keys(x)
    kc, ks = kc.cpu().numpy(), ks.cpu().numpy()
    assert np.array_equal(kc[50:50 + n], codes)
    assert np.array_equal(ks[50:50 + n].view(np.uint32), scales.view(np.uint32))
    assert np.all(kc[:50] == 0xAB) and np.all(kc[50 + n:] == 0xAB)  # nothing else written
    assert np.all(ks[:50] == -1.0) and np.all(ks[50 + n:] == -1.0)


def test_keys_slot_mapping():
    n, R = 3000, 5000
    x = _special_rows(n, 2)
    g = torch.Generator().manual_seed(3)
    slots = torch.randperm(R, generator=g)[:n].to(torch.int64)
    slots[::7] = -1                 # padding tokens: skipped
    slots[5::11] = R + 17           # past the cache: skipped
    kc = torch.zeros((R, 128), dtype=torch.uint8, device="cuda")
    ks = torch.full((R,), -1.0, dtype=torch.float32, device="cuda")
    ds4idx.quantize_keys(x.cuda(), kc, ks, slots=slots.cuda())
    torch.cuda.synchronize()
    codes, scales = _oracle_keys(x)
    kc, ks = kc.cpu().numpy(), ks.cpu().numpy()
    s = slots.numpy()
    ok = (s >= 0) & (s < R)
    assert np.array_equal(kc[s[ok]], codes[ok])
    assert np.array_equal(ks[s[ok]].view(np.uint32), scales[ok].view(np.uint32))
    untouched = np.setdiff1d(np.arange(R), s[ok])
    assert np.all(ks[untouched] == -1.0) and np.all(kc[untouched] == 0)


@pytest.mark.parametrize("in_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1, 333])
def test_queries_and_fold(in_dtype, T):
    g = torch.Generator().manual_seed(T)
    q = (torch.randn(T, 64, 128, generator=g) * torch.exp(torch.randn(T, 1, 1, generator=g) * 3))
    q[0, 3, :] = -0.0
    if T > 2:
        q[2] = 0.0  # whole token zero: scale 0, codes 0, w' = 0
    q = q.to(in_dtype)
    w = torch.randn(T, 64, generator=g) / 64
    qc, wo, qs = ds4idx.quantize_queries(q.cuda(), w.cuda())
    torch.cuda.synchronize()
    codes, scales = orc.quantize_rows(q.float().reshape(T, -1).numpy())
    assert np.array_equal(qc.cpu().numpy().reshape(T, -1), codes)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    wf = orc.fold_qscale(w.numpy(), scales)
    assert np.array_equal(wo.cpu().numpy().view(np.uint32), wf.view(np.uint32))
    # in place: w_out aliases w
    wd = w.cuda()
    ds4idx.quantize_queries(q.cuda(), wd, w_out=wd)
    torch.cuda.synchronize()
    assert np.array_equal(wd.cpu().numpy().view(np.uint32), wf.view(np.uint32))


@pytest.mark.parametrize("name", ["fp8_prefill_128k", "chunk_2048_at_260096"])
def test_workload_shapes(name):
    # The writer over a whole FP8 workload's fp32 draws reproduces the workload's codes, scales
    # and folded weights exactly; a row sample is also checked against the oracle directly.
    # (The 128k workload's 131072 query tokens would take 4 GiB of fp32 draws: its keys are
    # checked here, its queries have the same shape per token as the chunk's 2048.)
    spec = inputs.WORKLOADS[name]
    T, S, seed = spec["T"], spec["S"], spec["seed"]
    with_q = T <= 4096
    qf, kf, w = inputs.draw_f32(T, S, seed, parts=("q", "k", "w") if with_q else ("k",))
    prob_k, prob_ks = inputs.quantize_e4m3_rows(kf)
    kc = torch.empty((S, 128), dtype=torch.uint8, device="cuda")
    ks = torch.empty((S,), dtype=torch.float32, device="cuda")
    ds4idx.quantize_keys(kf.cuda(), kc, ks)
    if with_q:
        qc, wo, qs = ds4idx.quantize_queries(qf.cuda(), w.cuda())
    torch.cuda.synchronize()
    kc, ks = kc.cpu().numpy(), ks.cpu().numpy()
    assert np.array_equal(kc, prob_k.numpy())
    assert np.array_equal(ks.view(np.uint32), prob_ks.numpy().view(np.uint32))
    rows = np.random.default_rng(seed).integers(0, S, 4096)
    oc, os_ = orc.quantize_rows(kf.numpy()[rows])
    assert np.array_equal(kc[rows], oc) and np.array_equal(ks[rows], os_)
    if with_q:
        prob = inputs.workload(name)
        qcodes, qscale = orc.quantize_rows(qf.reshape(T, -1).numpy())
        assert np.array_equal(qc.cpu().numpy().reshape(T, -1), qcodes)
        assert np.array_equal(qc.cpu().numpy(), prob.q.numpy())
        assert np.array_equal(qs.cpu().numpy(), qscale)
        assert np.array_equal(wo.cpu().numpy(), orc.fold_qscale(w.numpy(), qscale))
        assert np.array_equal(wo.cpu().numpy(), prob.w.numpy())


def test_writer_rejects_bad_arguments():
    lib = ds4idx.load()
    x = torch.zeros(4, 128, device="cuda")
    kc = torch.zeros(4, 128, dtype=torch.uint8, device="cuda")
    ks = torch.zeros(4, device="cuda")
    P = lambda t: t.data_ptr()  # noqa: E731
    s = torch.cuda.current_stream().cuda_stream
    assert lib.ds4idx_quantize_keys(P(x), 1, 4, None, 0, P(kc), P(ks), 4, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_quantize_keys(P(x), 2, 4, None, 1, P(kc), P(ks), 4, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_quantize_keys(P(x) + 4, 2, 4, None, 0, P(kc), P(ks), 4, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_quantize_keys(None, 2, 4, None, 0, P(kc), P(ks), 4, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_quantize_keys(P(x), 2, 0, None, 0, P(kc), P(ks), 4, s) == ds4idx.OK
    assert lib.ds4idx_quantize_queries(None, 2, 4, None, None, None, None, s) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_quantize_queries(P(x), 7, 1, P(ks), P(kc), P(ks), None, s) == ds4idx.ERR_INVALID_ARG
