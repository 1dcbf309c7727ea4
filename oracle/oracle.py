"""ctypes front end of the fp64 Lightning Indexer oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's CPU-baseline leg call
this module; the product library never imports it. It shares no code with the CUDA path: it
takes raw input codes (bf16 bit patterns as uint16, OCP E4M3 bytes as uint8) plus fp32 arrays
as numpy buffers and decodes them itself.

What it computes (restated in ``oracle.cpp``): for each requested query row t, with
p = pos_offset + t, every key s <= min(p, S - 1) gets
``I[t,s] = kscale[s] * sum_j w[t,j] * max(0, q[t,j,:] . k[s,:])`` in fp64 (kscale = 1 for bf16),
and the top-k keeps the best min(topk, visible) keys ordered by score descending, ties to the
lower index, padded with (-1, -inf). Sources: "DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화"
(aitrends), sections 섹션별 상세 and 용어 해설; "DeepSeek V4 Flash는 단일 AMD MI300X에서
실행됩니다", section 두 가지 핵심 정확성 수정 사항 (FP8 indexer cache).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

BF16 = 0
FP8_E4M3 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``_build/liboracle.so`` (g++, OpenMP, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O3", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_scores.argtypes = [i32, p, p, p, p, i64, i64, i64, i64, i64, p, i64, p]
        lib.oracle_scores.restype = i32
        lib.oracle_topk.argtypes = [i32, p, p, p, p, i64, i64, i64, i64, i64, i64, p, i64, p, p]
        lib.oracle_topk.restype = i32
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_encode_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_encode_e4m3.restype = ctypes.c_uint8
        lib.oracle_quantize_rows.argtypes = [p, i64, i64, p, p]
        lib.oracle_quantize_rows.restype = i32
        lib.oracle_fold_qscale.argtypes = [p, p, i64, i64, p]
        lib.oracle_fold_qscale.restype = None
        lib.oracle_sparse_attention.argtypes = [p, p, i64, p, p, i64, i64, i64, i64, i64,
                                                ctypes.c_double, p, i64, p, p]
        lib.oracle_sparse_attention.restype = i32
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        _lib = lib
        return lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode_bf16(bits: int) -> float:
    return float(_load().oracle_decode_bf16(int(bits) & 0xFFFF))


def decode_e4m3(code: int) -> float:
    return float(_load().oracle_decode_e4m3(int(code) & 0xFF))


def _prep(dtype, q, w, k, kscale):
    code_t = np.uint16 if dtype == BF16 else np.uint8
    q = np.ascontiguousarray(q).view(code_t) if q.dtype != code_t else np.ascontiguousarray(q)
    k = np.ascontiguousarray(k).view(code_t) if k.dtype != code_t else np.ascontiguousarray(k)
    w = np.ascontiguousarray(w, dtype=np.float32)
    if q.ndim != 3 or k.ndim != 2 or w.ndim != 2:
        raise ValueError("expected q [T,H,D], w [T,H], k [S,D]")
    T, H, D = q.shape
    S = k.shape[0]
    if k.shape[1] != D or w.shape != (T, H):
        raise ValueError("shape mismatch between q, w and k")
    if dtype == FP8_E4M3:
        if kscale is None:
            raise ValueError("FP8 needs kscale")
        kscale = np.ascontiguousarray(kscale, dtype=np.float32)
        if kscale.shape != (S,):
            raise ValueError("kscale must be [S]")
    else:
        kscale = None
    return q, w, k, kscale, T, S, H, D


def _rows(rows, T):
    if rows is None:
        rows = np.arange(T, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def scores(dtype, q, w, k, kscale=None, pos_offset=0, rows=None) -> np.ndarray:
    """fp64 scores [len(rows), S]; entries past a row's causal limit are -inf."""
    q, w, k, kscale, T, S, H, D = _prep(dtype, q, w, k, kscale)
    rows = _rows(rows, T)
    out = np.empty((rows.shape[0], S), dtype=np.float64)
    rc = _load().oracle_scores(dtype, _ptr(q), _ptr(w), _ptr(k), _ptr(kscale), T, S, H, D,
                               int(pos_offset), _ptr(rows), rows.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError("oracle rejected the input (non-finite value, bad shape or row)")
    return out


def topk(dtype, q, w, k, kscale=None, pos_offset=0, topk=512, rows=None):
    """(idx int32 [n, topk], score fp64 [n, topk]) for the requested rows."""
    q, w, k, kscale, T, S, H, D = _prep(dtype, q, w, k, kscale)
    rows = _rows(rows, T)
    idx = np.empty((rows.shape[0], topk), dtype=np.int32)
    sc = np.empty((rows.shape[0], topk), dtype=np.float64)
    rc = _load().oracle_topk(dtype, _ptr(q), _ptr(w), _ptr(k), _ptr(kscale), T, S, H, D,
                             int(pos_offset), int(topk), _ptr(rows), rows.shape[0],
                             _ptr(idx), _ptr(sc))
    if rc != 0:
        raise ValueError("oracle rejected the input (non-finite value, bad shape or row)")
    return idx, sc


def select(score_rows: np.ndarray, n_visible: np.ndarray, topk: int):
    """The oracle's selection step alone, applied to given score rows.

    For each row r, the first n_visible[r] entries are ranked by (score descending, index
    ascending) and the first min(topk, n) kept, padded with (-1, nan-free -inf). Used to rerun the
    selection on scores the GPU emitted. Sorting is numpy's stable lexsort, a library primitive.
    """
    score_rows = np.asarray(score_rows)
    n_rows = score_rows.shape[0]
    idx = np.full((n_rows, topk), -1, dtype=np.int32)
    sc = np.full((n_rows, topk), -np.inf, dtype=score_rows.dtype)
    for r in range(n_rows):
        n = int(n_visible[r])
        row = score_rows[r, :n]
        # Treat -0.0 and +0.0 as equal, as numeric comparison does.
        keyrow = np.where(row == 0, 0, row)
        order = np.lexsort((np.arange(n), -keyrow.astype(np.float64)))
        m = min(topk, n)
        idx[r, :m] = order[:m]
        sc[r, :m] = row[order[:m]]
    return idx, sc


# ---------------------------------------------------------------- FP8 index-cache writer

def encode_e4m3(y: float) -> int:
    """Nearest OCP E4M3FN code (ties to the even code, saturating at 448, sign kept)."""
    return int(_load().oracle_encode_e4m3(float(y)))


def quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-row absmax/448 E4M3 quantisation of x [R, C] fp32 -> (codes u8 [R, C], scale f32 [R]).

    scale = fp32(absmax / 448); code = E4M3(clamp(fp32(x / scale), +-448)); scale 0 -> codes 0.
    ("DeepSeek V4 Flash는 단일 AMD MI300X에서 실행됩니다", FP8 형식 불일치: the FP8 indexer cache.)
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("expected x [R, C]")
    R, C = x.shape
    codes = np.empty((R, C), dtype=np.uint8)
    scales = np.empty((R,), dtype=np.float32)
    if _load().oracle_quantize_rows(_ptr(x), R, C, _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("oracle rejected the input (non-finite value or bad shape)")
    return codes, scales


def fold_qscale(w, qscale) -> np.ndarray:
    """w' [T, H] = fp32(w * qscale[t]) (the query scale folded into the head weights)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    qscale = np.ascontiguousarray(qscale, dtype=np.float32)
    T, H = w.shape
    if qscale.shape != (T,):
        raise ValueError("qscale must be [T]")
    out = np.empty_like(w)
    _load().oracle_fold_qscale(_ptr(w), _ptr(qscale), T, H, _ptr(out))
    return out


# ---------------------------------------------------------------- sparse attention

def sparse_attention(q, kv, idx, scale, d_v, row0=None, rows=None):
    """fp64 sparse attention over the selected keys (``oracle.cpp``): q [T, H, Dqk] and kv
    [R, Dqk] as bf16 codes (uint16) or torch bf16, idx [T, K] int32 key positions (-1 empty),
    row0 [T] int64 kv row of key 0 per token (None: 0). Returns (out [n, H, d_v], lse [n, H]).
    ("DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화", 용어 해설: 희소 어텐션.)"""
    def codes(a):
        if hasattr(a, "view") and str(getattr(a, "dtype", "")) == "torch.bfloat16":
            a = a.view(__import__("torch").int16).numpy()
        return np.ascontiguousarray(np.asarray(a)).view(np.uint16)
    q, kv = codes(q), codes(kv)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, H, Dqk = q.shape
    R = kv.shape[0]
    K = idx.shape[1]
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    r0 = None if row0 is None else np.ascontiguousarray(row0, dtype=np.int64)
    out = np.empty((rows.shape[0], H, d_v), dtype=np.float64)
    lse = np.empty((rows.shape[0], H), dtype=np.float64)
    rc = _load().oracle_sparse_attention(_ptr(q), _ptr(kv), R, _ptr(idx), _ptr(r0), T, H, Dqk,
                                         d_v, K, float(scale), _ptr(rows), rows.shape[0],
                                         _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle rejected the input")
    return out, lse
