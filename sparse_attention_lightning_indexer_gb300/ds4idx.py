"""Python binding of the ds4idx C ABI (include/ds4idx.h): argument marshalling only.

Every step of the indexer runs in the CUDA kernels of ``libds4idx.so``; this module checks
tensor shapes, dtypes and devices, passes raw device pointers and the current CUDA stream, and
turns status codes into exceptions. PyTorch provides device memory and streams. There is no
CPU fallback: if the library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

BF16 = 0
FP8_E4M3 = 1
F32 = 2
H_I = 64
D_I = 128
TOPK = 512

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_ALLOC = -3
ERR_LAUNCH = -4
ERR_DEVICE_TIMEOUT = -5
ERR_CUDA = -6
ERR_SCRATCH_LIMIT = -7

EXPORTS = ("ds4idx_create", "ds4idx_score_topk", "ds4idx_score_topk_batched",
           "ds4idx_score_dense_debug", "ds4idx_sync_status", "ds4idx_destroy",
           "ds4idx_status_string", "ds4idx_version", "ds4idx_score_topk_batched_noalloc",
           "ds4idx_kernels_launched", "ds4idx_debug_wait_test", "ds4idx_plan_query",
           "ds4idx_quantize_keys", "ds4idx_quantize_queries", "ds4idx_score_topk_varlen",
           "ds4idx_merge_topk", "ds4idx_sparse_attention", "ds4idx_sparse_attention_status")

_lock = threading.Lock()
_lib = None


class Ds4IdxError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("max_T", ctypes.c_int64), ("max_S", ctypes.c_int64),
                ("max_batch", ctypes.c_int64)]


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Loads libds4idx.so (built in-tree by ``build.build()``). Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(f"ds4idx library not built: {p} is missing (run build())")
        lib = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.ds4idx_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(Config)]
        lib.ds4idx_create.restype = ctypes.c_int
        lib.ds4idx_score_topk.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp, vp]
        lib.ds4idx_score_topk.restype = ctypes.c_int
        lib.ds4idx_score_topk_batched.argtypes = [vp, i32, vp, vp, vp, vp, i64, i64, vp, i32, vp,
                                                  vp, vp]
        lib.ds4idx_score_topk_batched.restype = ctypes.c_int
        lib.ds4idx_score_dense_debug.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp, vp]
        lib.ds4idx_score_dense_debug.restype = ctypes.c_int
        lib.ds4idx_sync_status.argtypes = [vp, vp]
        lib.ds4idx_sync_status.restype = ctypes.c_int
        lib.ds4idx_destroy.argtypes = [vp]
        lib.ds4idx_destroy.restype = ctypes.c_int
        lib.ds4idx_status_string.argtypes = [ctypes.c_int]
        lib.ds4idx_status_string.restype = ctypes.c_char_p
        lib.ds4idx_version.argtypes = []
        lib.ds4idx_version.restype = ctypes.c_int
        lib.ds4idx_score_topk_batched_noalloc.argtypes = [i32, i32, vp, vp, vp, vp, i64, i64, vp,
                                                          i32, vp, vp, vp]
        lib.ds4idx_score_topk_batched_noalloc.restype = ctypes.c_int
        lib.ds4idx_kernels_launched.argtypes = []
        lib.ds4idx_kernels_launched.restype = ctypes.c_uint64
        lib.ds4idx_debug_wait_test.argtypes = [vp, ctypes.c_uint64, i32]
        lib.ds4idx_debug_wait_test.restype = ctypes.c_int
        lib.ds4idx_plan_query.argtypes = [i32, i32, i64, i64, vp, i32, vp]
        lib.ds4idx_plan_query.restype = ctypes.c_int
        lib.ds4idx_score_topk_varlen.argtypes = [vp, i32, vp, vp, vp, vp, vp, i64, vp, vp, i32,
                                                 i32, vp, vp, i32, vp, vp, vp]
        lib.ds4idx_score_topk_varlen.restype = ctypes.c_int
        lib.ds4idx_sparse_attention.argtypes = [vp, vp, i64, vp, vp, i64, i32, i32, i32, i32,
                                                ctypes.c_float, vp, vp, vp]
        lib.ds4idx_sparse_attention.restype = ctypes.c_int
        lib.ds4idx_sparse_attention_status.argtypes = [vp]
        lib.ds4idx_sparse_attention_status.restype = ctypes.c_int
        lib.ds4idx_merge_topk.argtypes = [i32, i64, vp, vp, vp, vp, i32, vp, vp, vp]
        lib.ds4idx_merge_topk.restype = ctypes.c_int
        lib.ds4idx_quantize_keys.argtypes = [vp, i32, i64, vp, i64, vp, vp, i64, vp]
        lib.ds4idx_quantize_keys.restype = ctypes.c_int
        lib.ds4idx_quantize_queries.argtypes = [vp, i32, i64, vp, vp, vp, vp, vp]
        lib.ds4idx_quantize_queries.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def kernels_launched() -> int:
    """Kernels the library has enqueued in this process (its own count, for benchmarks)."""
    return int(load().ds4idx_kernels_launched())


PLAN_FIELDS = ("queries_per_cta", "query_blocks", "splits", "tiles_per_split", "grid",
               "list_words", "tickets")


def plan_query(num_sms: int, B: int, T: int, S: int, pos_offsets, fixed_scratch: bool = False):
    """The work decomposition of a call (host computation only): a dict of PLAN_FIELDS."""
    pos = (ctypes.c_int64 * B)(*[int(x) for x in pos_offsets])
    out = (ctypes.c_int64 * len(PLAN_FIELDS))()
    _check(load().ds4idx_plan_query(num_sms, B, T, S, ctypes.cast(pos, ctypes.c_void_p),
                                    1 if fixed_scratch else 0, ctypes.cast(out, ctypes.c_void_p)),
           "ds4idx_plan_query")
    return dict(zip(PLAN_FIELDS, list(out)))


def _in_dtype(t: torch.Tensor, name: str) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"{name} must be float32 or bfloat16")


def quantize_keys(k, kcache, kscale, dst_offset: int = 0, slots=None, stream=None):
    """Writes k [n, 128] (fp32/bf16) as E4M3 codes + scales into kcache [R, 128] uint8 /
    kscale [R] fp32, at rows dst_offset.. or at slots [n] (int64, -1 skips a row)."""
    n = k.shape[0]
    _need(k, (n, D_I), "k")
    R = kcache.shape[0]
    _need(kcache, (R, D_I), "kcache", torch.uint8)
    _need(kscale, (R,), "kscale", torch.float32)
    if slots is not None:
        _need(slots, (n,), "slots", torch.int64)
    _check(load().ds4idx_quantize_keys(_ptr(k), _in_dtype(k, "k"), n, _ptr(slots),
                                       int(dst_offset), _ptr(kcache), _ptr(kscale), R,
                                       _stream_ptr(stream)), "ds4idx_quantize_keys")
    return kcache, kscale


def quantize_queries(q, w, q_codes=None, w_out=None, qscale=None, stream=None):
    """q [T, 64, 128] (fp32/bf16), w [T, 64] -> (E4M3 codes [T, 64, 128] uint8, w' [T, 64],
    qscale [T])."""
    T = q.shape[0]
    _need(q, (T, H_I, D_I), "q")
    _need(w, (T, H_I), "w", torch.float32)
    dev = q.device
    if q_codes is None:
        q_codes = torch.empty((T, H_I, D_I), dtype=torch.uint8, device=dev)
    if w_out is None:
        w_out = torch.empty((T, H_I), dtype=torch.float32, device=dev)
    if qscale is None:
        qscale = torch.empty((T,), dtype=torch.float32, device=dev)
    _need(q_codes, (T, H_I, D_I), "q_codes", torch.uint8)
    _need(w_out, (T, H_I), "w_out", torch.float32)
    _need(qscale, (T,), "qscale", torch.float32)
    _check(load().ds4idx_quantize_queries(_ptr(q), _in_dtype(q, "q"), T, _ptr(w), _ptr(q_codes),
                                          _ptr(w_out), _ptr(qscale), _stream_ptr(stream)),
           "ds4idx_quantize_queries")
    return q_codes, w_out, qscale


def merge_topk(in_idx, in_score, idx_offsets, row0=None, out_idx=None, out_score=None,
               stream=None):
    """Merges key-sharded Top-512 lists: in_idx / in_score [L, rows, 512] (shard-local indices,
    -1 empty), idx_offsets: L host ints (each shard's first key), row0: L host ints or None.
    Returns (out_idx [rows, 512], out_score [rows, 512])."""
    L, rows = in_idx.shape[0], in_idx.shape[1]
    _need(in_idx, (L, rows, TOPK), "in_idx", torch.int32)
    _need(in_score, (L, rows, TOPK), "in_score", torch.float32)
    dev = in_idx.device
    if out_idx is None:
        out_idx = torch.empty((rows, TOPK), dtype=torch.int32, device=dev)
    if out_score is None:
        out_score = torch.empty((rows, TOPK), dtype=torch.float32, device=dev)
    _need(out_idx, (rows, TOPK), "out_idx", torch.int32)
    _need(out_score, (rows, TOPK), "out_score", torch.float32)
    if len(idx_offsets) != L or (row0 is not None and len(row0) != L):
        raise ValueError("idx_offsets and row0 need one entry per list")
    offs = (ctypes.c_int64 * L)(*[int(x) for x in idx_offsets])
    r0 = None if row0 is None else (ctypes.c_int64 * L)(*[int(x) for x in row0])
    vp = ctypes.c_void_p
    _check(load().ds4idx_merge_topk(L, rows, _ptr(in_idx), _ptr(in_score), ctypes.cast(offs, vp),
                                    None if r0 is None else ctypes.cast(r0, vp), TOPK,
                                    _ptr(out_idx), _ptr(out_score), _stream_ptr(stream)),
           "ds4idx_merge_topk")
    return out_idx, out_score


SA_HEADS, SA_DQK, SA_DV = 128, 576, 512


def sparse_attention(q, kv, idx, sm_scale: float, kv_row0=None, out=None, lse=None, stream=None):
    """Attention of q [T, 128, 576] (bf16) over the selected rows of kv [R, 576] (bf16):
    idx [T, 512] int32 positions (-1 empty), kv_row0 [T] int64 or None.
    Returns (out [T, 128, 512] bf16, lse [T, 128] fp32)."""
    T, R = q.shape[0], kv.shape[0]
    _need(q, (T, SA_HEADS, SA_DQK), "q", torch.bfloat16)
    _need(kv, (R, SA_DQK), "kv", torch.bfloat16)
    _need(idx, (T, TOPK), "idx", torch.int32)
    if kv_row0 is not None:
        _need(kv_row0, (T,), "kv_row0", torch.int64)
    if out is None:
        out = torch.empty((T, SA_HEADS, SA_DV), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, SA_HEADS), dtype=torch.float32, device=q.device)
    _need(out, (T, SA_HEADS, SA_DV), "out", torch.bfloat16)
    _need(lse, (T, SA_HEADS), "lse", torch.float32)
    _check(load().ds4idx_sparse_attention(_ptr(q), _ptr(kv), R, _ptr(idx), _ptr(kv_row0), T,
                                          SA_HEADS, SA_DQK, SA_DV, TOPK, float(sm_scale),
                                          _ptr(out), _ptr(lse), _stream_ptr(stream)),
           "ds4idx_sparse_attention")
    return out, lse


def sparse_attention_status(stream=None):
    _check(load().ds4idx_sparse_attention_status(_stream_ptr(stream)), "ds4idx_sparse_attention")


def status_string(status: int) -> str:
    try:
        return load().ds4idx_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(status: int, what: str):
    if status != OK:
        raise Ds4IdxError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _codes(t: torch.Tensor, dtype: int, name: str) -> torch.Tensor:
    if dtype == BF16:
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16 for a bf16 indexer")
        return t
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8)
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must be float8_e4m3fn or uint8 E4M3 codes for an FP8 indexer")
    return t


def _need(t: torch.Tensor, shape, name: str, dtype=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}")


class Indexer:
    """One ds4idx handle (device workspace) for a dtype and maximum sizes."""

    def __init__(self, dtype: int = BF16, max_T: int = 65536, max_S: int = 65536,
                 max_batch: int = 1, n_heads: int = H_I, head_dim: int = D_I, topk: int = TOPK):
        self._lib = load()
        self.dtype = dtype
        self.topk = topk
        cfg = Config(n_heads, head_dim, topk, dtype, max_T, max_S, max_batch)
        h = ctypes.c_void_p()
        _check(self._lib.ds4idx_create(ctypes.byref(h), ctypes.byref(cfg)), "ds4idx_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.ds4idx_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def score_topk(self, q, w, kcache, kscale=None, pos_offset: int = 0, out_idx=None,
                   out_score=None, stream=None, want_score: bool = True):
        """q [T,64,128], w [T,64] fp32, kcache [S,128], kscale [S] fp32 (FP8) -> (idx, score)."""
        T, S = q.shape[0], kcache.shape[0]
        q = _codes(q, self.dtype, "q")
        kcache = _codes(kcache, self.dtype, "kcache")
        _need(q, (T, H_I, D_I), "q")
        _need(w, (T, H_I), "w", torch.float32)
        _need(kcache, (S, D_I), "kcache")
        if kscale is not None:
            _need(kscale, (S,), "kscale", torch.float32)
        dev = q.device
        if out_idx is None:
            out_idx = torch.empty((T, self.topk), dtype=torch.int32, device=dev)
        if out_score is None and want_score:
            out_score = torch.empty((T, self.topk), dtype=torch.float32, device=dev)
        _need(out_idx, (T, self.topk), "out_idx", torch.int32)
        if out_score is not None:
            _need(out_score, (T, self.topk), "out_score", torch.float32)
        st = self._lib.ds4idx_score_topk(self._h, _ptr(q), _ptr(w), _ptr(kcache), _ptr(kscale),
                                         T, S, int(pos_offset), self.topk, _ptr(out_idx),
                                         _ptr(out_score), _stream_ptr(stream))
        _check(st, "ds4idx_score_topk")
        return out_idx, out_score

    def score_topk_batched(self, q, w, kcache, kscale, pos_offsets, out_idx=None, out_score=None,
                           stream=None):
        """q [B,T,64,128], w [B,T,64], kcache [B,S,128], kscale [B,S]; pos_offsets: B ints."""
        B, T, S = q.shape[0], q.shape[1], kcache.shape[1]
        q = _codes(q, self.dtype, "q")
        kcache = _codes(kcache, self.dtype, "kcache")
        _need(q, (B, T, H_I, D_I), "q")
        _need(w, (B, T, H_I), "w", torch.float32)
        _need(kcache, (B, S, D_I), "kcache")
        if kscale is not None:
            _need(kscale, (B, S), "kscale", torch.float32)
        dev = q.device
        if out_idx is None:
            out_idx = torch.empty((B, T, self.topk), dtype=torch.int32, device=dev)
        if out_score is None:
            out_score = torch.empty((B, T, self.topk), dtype=torch.float32, device=dev)
        _need(out_idx, (B, T, self.topk), "out_idx", torch.int32)
        _need(out_score, (B, T, self.topk), "out_score", torch.float32)
        pos = (ctypes.c_int64 * B)(*[int(x) for x in pos_offsets])
        st = self._lib.ds4idx_score_topk_batched(self._h, B, _ptr(q), _ptr(w), _ptr(kcache),
                                                 _ptr(kscale), T, S, ctypes.cast(pos, ctypes.c_void_p),
                                                 self.topk, _ptr(out_idx), _ptr(out_score),
                                                 _stream_ptr(stream))
        _check(st, "ds4idx_score_topk_batched")
        return out_idx, out_score

    def score_topk_varlen(self, q, w, cu_seqlens_q, kcache, kscale, seq_lens, pos_offsets,
                          kv_start=None, page_table=None, page_size: int = 0, out_idx=None,
                          out_score=None, stream=None):
        """Sequences of different lengths in one launch (see include/ds4idx.h).

        q [Q, 64, 128], w [Q, 64]: packed queries, sequence b owning rows
        cu_seqlens_q[b]..cu_seqlens_q[b+1]-1 (host ints, B + 1 of them). kcache [R, 128] (+ kscale
        [R]) is the key pool: sequence b's keys start at pool row kv_start[b], or are found through
        page_table [B, P] (int32, on the device) with page_size keys per page.
        seq_lens, pos_offsets: B host ints. Returns (out_idx, out_score), [Q, topk].
        """
        B = len(seq_lens)
        Q, R = q.shape[0], kcache.shape[0]
        q = _codes(q, self.dtype, "q")
        kcache = _codes(kcache, self.dtype, "kcache")
        _need(q, (Q, H_I, D_I), "q")
        _need(w, (Q, H_I), "w", torch.float32)
        _need(kcache, (R, D_I), "kcache")
        if kscale is not None:
            _need(kscale, (R,), "kscale", torch.float32)
        if len(cu_seqlens_q) != B + 1 or len(pos_offsets) != B:
            raise ValueError("cu_seqlens_q needs B + 1 entries and pos_offsets B")
        if page_table is not None:
            _need(page_table, tuple(page_table.shape), "page_table", torch.int32)
            if page_table.dim() != 2 or page_table.shape[0] != B:
                raise ValueError("page_table must be [B, pages_per_seq]")
        dev = q.device
        if out_idx is None:
            out_idx = torch.empty((Q, self.topk), dtype=torch.int32, device=dev)
        if out_score is None:
            out_score = torch.empty((Q, self.topk), dtype=torch.float32, device=dev)
        _need(out_idx, (Q, self.topk), "out_idx", torch.int32)
        _need(out_score, (Q, self.topk), "out_score", torch.float32)
        I64 = ctypes.c_int64
        cu = (I64 * (B + 1))(*[int(x) for x in cu_seqlens_q])
        sl = (I64 * B)(*[int(x) for x in seq_lens])
        po = (I64 * B)(*[int(x) for x in pos_offsets])
        ks = None if kv_start is None else (I64 * B)(*[int(x) for x in kv_start])
        vp = ctypes.c_void_p
        st = self._lib.ds4idx_score_topk_varlen(
            self._h, B, _ptr(q), _ptr(w), ctypes.cast(cu, vp), _ptr(kcache), _ptr(kscale), R,
            None if ks is None else ctypes.cast(ks, vp), _ptr(page_table), int(page_size),
            0 if page_table is None else int(page_table.shape[1]), ctypes.cast(sl, vp),
            ctypes.cast(po, vp), self.topk, _ptr(out_idx), _ptr(out_score), _stream_ptr(stream))
        _check(st, "ds4idx_score_topk_varlen")
        return out_idx, out_score

    def score_dense_debug(self, q, w, kcache, kscale=None, pos_offset: int = 0, out=None,
                          stream=None):
        """fp32 scores [T, S] as the selection kernels see them (-inf where not visible)."""
        T, S = q.shape[0], kcache.shape[0]
        q = _codes(q, self.dtype, "q")
        kcache = _codes(kcache, self.dtype, "kcache")
        _need(q, (T, H_I, D_I), "q")
        _need(w, (T, H_I), "w", torch.float32)
        _need(kcache, (S, D_I), "kcache")
        if kscale is not None:
            _need(kscale, (S,), "kscale", torch.float32)
        if out is None:
            out = torch.empty((T, S), dtype=torch.float32, device=q.device)
        _need(out, (T, S), "out", torch.float32)
        st = self._lib.ds4idx_score_dense_debug(self._h, _ptr(q), _ptr(w), _ptr(kcache),
                                                _ptr(kscale), T, S, int(pos_offset), _ptr(out),
                                                _stream_ptr(stream))
        _check(st, "ds4idx_score_dense_debug")
        return out

    def debug_wait_test(self, wait_limit_ns: int = 2_000_000_000, withhold: bool = False):
        """Test support: bounded-wait limit for later calls, and one withheld arrival."""
        _check(self._lib.ds4idx_debug_wait_test(self._h, int(wait_limit_ns), 1 if withhold else 0),
               "ds4idx_debug_wait_test")

    def sync_status(self, stream=None):
        _check(self._lib.ds4idx_sync_status(self._h, _stream_ptr(stream)), "ds4idx_sync_status")
