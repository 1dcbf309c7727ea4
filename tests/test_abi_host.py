"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a, loads, exports
every entry point include/ds4idx.h declares, and rejects bad arguments before any device work.
"""
import ctypes
import os
import re

import pytest
import torch

from sparse_attention_lightning_indexer_gb300 import build, ds4idx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds4idx.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ds4idx.load()


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|uint64_t|const char\s*\*)\s+(ds4idx_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ("ds4idx_create", "ds4idx_score_topk", "ds4idx_score_topk_batched",
              "ds4idx_score_dense_debug", "ds4idx_destroy", "ds4idx_status_string"):
        assert n in names
    assert set(names) == set(ds4idx.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for n in declared():
        assert hasattr(lib, n), f"{n} not exported by {ds4idx.library_path()}"


def test_status_strings_and_version(lib):
    for code in range(0, -8, -1):
        s = lib.ds4idx_status_string(code).decode()
        assert s and s != "unknown status", code
    assert lib.ds4idx_status_string(-99).decode() == "unknown status"
    assert lib.ds4idx_version() == (1 << 16) | 1
    assert lib.ds4idx_kernels_launched() == 0  # nothing launched without a device


def _cfg(**kw):
    base = dict(n_heads=64, head_dim=128, topk=512, dtype=0, max_T=128, max_S=1024, max_batch=1)
    base.update(kw)
    return ds4idx.Config(**base)


def test_create_validates_before_touching_the_device(lib):
    h = ctypes.c_void_p(1234)
    assert lib.ds4idx_create(None, ctypes.byref(_cfg())) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_create(ctypes.byref(h), None) == ds4idx.ERR_INVALID_ARG
    assert h.value is None  # *out is cleared on error
    for bad in (dict(dtype=7), dict(max_T=0), dict(max_S=0), dict(max_batch=0),
                dict(max_batch=65), dict(max_S=1 << 31)):
        assert lib.ds4idx_create(ctypes.byref(h), ctypes.byref(_cfg(**bad))) == \
            ds4idx.ERR_INVALID_ARG, bad
    for bad in (dict(n_heads=32), dict(head_dim=64), dict(topk=2048)):
        assert lib.ds4idx_create(ctypes.byref(h), ctypes.byref(_cfg(**bad))) == \
            ds4idx.ERR_UNSUPPORTED, bad


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_create_without_a_device_reports_cuda_error(lib):
    h = ctypes.c_void_p()
    assert lib.ds4idx_create(ctypes.byref(h), ctypes.byref(_cfg())) == ds4idx.ERR_CUDA
    assert h.value is None


def test_null_handle_and_bad_arguments(lib):
    assert lib.ds4idx_score_topk(None, None, None, None, None, 4, 16, 0, 512, None, None,
                                 None) == ds4idx.ERR_INVALID_ARG
    pos = (ctypes.c_int64 * 1)(0)
    assert lib.ds4idx_score_topk_batched(None, 1, None, None, None, None, 4, 16,
                                         ctypes.cast(pos, ctypes.c_void_p), 512, None, None,
                                         None) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_score_dense_debug(None, None, None, None, None, 4, 16, 0, None,
                                        None) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_sync_status(None, None) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_destroy(None) == ds4idx.OK
    # no-allocation entry: argument errors are found before any device call
    p = ctypes.cast(pos, ctypes.c_void_p)
    assert lib.ds4idx_score_topk_batched_noalloc(9, 1, None, None, None, None, 4, 16, p, 512,
                                                 None, None, None) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_score_topk_batched_noalloc(0, 0, None, None, None, None, 4, 16, p, 512,
                                                 None, None, None) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_score_topk_batched_noalloc(0, 1, None, None, None, None, 4, 16, None, 512,
                                                 None, None, None) == ds4idx.ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        ds4idx.load(str(tmp_path / "missing.so"))


# ---- work decomposition (host arithmetic only, for the 152-SM GB300)

def _plan(lib, B, T, S, pos, fixed=False, sms=152):
    return ds4idx.plan_query(sms, B, T, S, pos, fixed_scratch=fixed)


def test_plans_of_the_workloads(lib):
    p = _plan(lib, 1, 65536, 65536, [0])  # prefill: query blocks alone fill the GPU
    assert (p["queries_per_cta"], p["query_blocks"], p["splits"], p["grid"]) == (4, 16384, 1, 16384)
    assert p["list_words"] == 0 and p["tickets"] == 0
    p = _plan(lib, 8, 1, 262144, [262143] * 8)  # decode: 19 splits x 8 sequences = one wave
    assert (p["queries_per_cta"], p["splits"], p["grid"]) == (1, 19, 152)
    assert p["list_words"] == 8 * 19 * 1152 and p["tickets"] == 8
    p = _plan(lib, 1, 2048, 262144, [260096])  # the 2048-token chunk: two splits
    assert (p["splits"], p["grid"], p["list_words"]) == (2, 1024, 1 << 21)


def test_fixed_scratch_plans_fit_and_match_when_possible(lib):
    # The handle plan splits a 768-token chunk further than the fixed array holds.
    h = _plan(lib, 1, 768, 262144, [262144 - 768])
    assert h["list_words"] > 1 << 21
    f = _plan(lib, 1, 768, 262144, [262144 - 768], fixed=True)
    assert 1 < f["splits"] < h["splits"] and f["list_words"] <= 1 << 21
    # Where the handle plan fits, the fixed-scratch plan is the same plan.
    for args in ((8, 1, 262144, [262143] * 8), (1, 2048, 262144, [260096]),
                 (4, 6, 5000, [4994, 1200, 0, 7])):
        assert _plan(lib, *args) == _plan(lib, *args, fixed=True)
    # Every fixed-scratch plan fits, whatever the shape.
    for B in (1, 2, 8, 64):
        for T in (1, 2, 5, 64, 700, 1100, 2100, 4096):
            for S in (1, 600, 9000, 262144, 1 << 20, (1 << 31) - 1):
                pos = [max(0, S - T)] * B
                f = _plan(lib, B, T, S, pos, fixed=True)
                assert f["list_words"] <= 1 << 21 and f["tickets"] <= 4096, (B, T, S, f)
                assert f["grid"] == B * f["query_blocks"] * f["splits"]


def test_plan_query_rejects_bad_arguments(lib):
    out = (ctypes.c_int64 * 7)()
    pos = (ctypes.c_int64 * 1)(0)
    p = ctypes.cast(pos, ctypes.c_void_p)
    o = ctypes.cast(out, ctypes.c_void_p)
    assert lib.ds4idx_plan_query(0, 1, 1, 16, p, 0, o) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_plan_query(152, 65, 1, 16, p, 0, o) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_plan_query(152, 1, 0, 16, p, 0, o) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_plan_query(152, 1, 1, 16, None, 0, o) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_plan_query(152, 1, 1, 16, p, 0, None) == ds4idx.ERR_INVALID_ARG
    assert lib.ds4idx_debug_wait_test(None, 2000000000, 0) == ds4idx.ERR_INVALID_ARG
