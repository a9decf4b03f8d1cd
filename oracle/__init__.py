"""CPU fp64 oracle for single-token MLA decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product library never loads it and shares no code
with it.  The arithmetic lives in ``mla_oracle.c`` (plain C, fp64, optional OpenMP
over batch rows); this module compiles it with gcc on first use and calls it through
ctypes with host (CPU) buffers.

Functions and what pins each one (see ``tests/test_oracle.py``):

* ``e4m3`` / ``e2m1`` / ``e8m0`` / ``bf16`` decoders -- exhaustive code tables against
  PyTorch's own float8 / e8m0 / bf16 conversions and against the OCP MX e2m1 value table.
* ``attend`` / ``decode`` -- closed forms (one cached token returns its V; identical keys
  or q = 0 return the mean of V; a constant V column is returned unchanged; exact
  two-token logits through a rope feature), the log-sum-exp closed form, brute force on
  tiny inputs, cross-encoding consistency (fp8 / MXFP4 caches vs the bf16 cache holding
  their decoded values) and the pages' 0.1/0.1 quantisation tolerance.
* ``combine`` -- the merge of per-range partial results reproduces the full-range result.
* ``split_range`` -- the ranges of all splits tile [0, L) in BN-rounded chunks.
* ``paged_rows`` / ``decode_paged`` -- a hand-written page table's row lists; an identity
  page table reproduces the contiguous decode; a shuffled one gives the same result as
  the contiguous cache it was built from.
* ``decode_paged_multi`` -- one token per sequence reproduces ``decode_paged``; each query
  row of a hand-built two-token case equals the decode of its own hand-cut prefix; a first
  query token that sees one cached token returns that token's value.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

NH, D, DV = 16, 576, 512
KV_BF16, KV_FP8, KV_MXFP4 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into a shared library (gcc -O2 -fopenmp)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dbl, vp, i64, c_int = ctypes.c_double, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        for name in ("mla_oracle_e4m3", "mla_oracle_e2m1", "mla_oracle_e8m0"):
            getattr(lib, name).restype = dbl
            getattr(lib, name).argtypes = [c_int]
        lib.mla_oracle_bf16.restype = dbl
        lib.mla_oracle_bf16.argtypes = [ctypes.c_uint16]
        lib.mla_oracle_dequant_row.restype = None
        lib.mla_oracle_dequant_row.argtypes = [c_int, vp, vp, i64, vp]
        lib.mla_oracle_attend.restype = c_int
        lib.mla_oracle_attend.argtypes = [vp, c_int, vp, vp, i64, i64, vp, vp]
        lib.mla_oracle_decode.restype = c_int
        lib.mla_oracle_decode.argtypes = [vp, c_int, vp, vp, vp, c_int, vp, vp, c_int]
        lib.mla_oracle_combine.restype = None
        lib.mla_oracle_combine.argtypes = [c_int, vp, vp, vp, vp]
        lib.mla_oracle_split_range.restype = None
        lib.mla_oracle_split_range.argtypes = [i64, c_int, c_int, c_int,
                                               ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.mla_oracle_max_threads.restype = c_int
        lib.mla_oracle_max_threads.argtypes = []
        _lib = lib
        return lib


def _np(x, dtype=None):
    """torch tensor / numpy array -> contiguous host numpy array (no arithmetic)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        x = t.numpy()
    a = np.ascontiguousarray(x)
    if dtype is not None:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e4m3(code: int) -> float:
    return _load().mla_oracle_e4m3(int(code))


def e2m1(code: int) -> float:
    return _load().mla_oracle_e2m1(int(code))


def e8m0(code: int) -> float:
    return _load().mla_oracle_e8m0(int(code))


def bf16(bits: int) -> float:
    return _load().mla_oracle_bf16(int(bits) & 0xFFFF)


def _kv_args(kv, kv_scale, kv_dtype):
    if kv_dtype == KV_BF16:
        return _np(kv, np.uint16), None
    if kv_dtype == KV_FP8:
        return _np(kv, np.uint8), _np(kv_scale, np.float32)
    if kv_dtype == KV_MXFP4:
        return _np(kv, np.uint8), _np(kv_scale, np.uint8)
    raise ValueError(kv_dtype)


def dequant_rows(kv, kv_scale, kv_dtype, rows) -> np.ndarray:
    """Decoded rows (fp64 [len(rows), 576])."""
    lib = _load()
    k, s = _kv_args(kv, kv_scale, kv_dtype)
    out = np.zeros((len(rows), D), dtype=np.float64)
    for i, r in enumerate(rows):
        lib.mla_oracle_dequant_row(kv_dtype, _ptr(k), _ptr(s), int(r), _ptr(out[i]))
    return out


def attend(q_b, kv, kv_scale, kv_dtype, r0: int, r1: int):
    """One batch row (q_b: bf16 [16, 576]) over cached rows [r0, r1) ->
    (o fp64 [16, 512], lse fp64 [16])."""
    lib = _load()
    qa = _np(q_b, np.uint16).reshape(NH, D)
    k, s = _kv_args(kv, kv_scale, kv_dtype)
    o = np.zeros((NH, DV), dtype=np.float64)
    lse = np.zeros((NH,), dtype=np.float64)
    rc = lib.mla_oracle_attend(_ptr(qa), kv_dtype, _ptr(k), _ptr(s), int(r0), int(r1), _ptr(o), _ptr(lse))
    if rc:
        raise MemoryError("oracle attend failed")
    return o, lse


def decode(q, kv, kv_scale, kv_indptr, kv_dtype, nthreads: int = 0):
    """Whole decode -> (out fp64 [B, 16, 512], lse fp64 [B, 16])."""
    lib = _load()
    qa = _np(q, np.uint16)
    B = qa.shape[0]
    k, s = _kv_args(kv, kv_scale, kv_dtype)
    ip = _np(kv_indptr, np.int32)
    out = np.zeros((B, NH, DV), dtype=np.float64)
    lse = np.zeros((B, NH), dtype=np.float64)
    rc = lib.mla_oracle_decode(_ptr(qa), kv_dtype, _ptr(k), _ptr(s), _ptr(ip), B, _ptr(out), _ptr(lse),
                               int(nthreads))
    if rc:
        raise MemoryError("oracle decode failed")
    return out, lse


def paged_rows(page_indptr, page_indices, last_page_len, page_size: int):
    """Physical cache rows of every sequence of a paged cache, in token order.

    The page table of the paged MLA decode interface (amd-mixed-mla submission 700955,
    `_get_a16w8_persistent_state`: a page-level kv_indptr, kv_indices and kv_last_page_len
    for a given page_size): sequence b owns the pages
    page_indices[page_indptr[b] : page_indptr[b+1]], all full except the last, which holds
    last_page_len[b] tokens.  Token t of sequence b therefore lives at physical row
    page_indices[page_indptr[b] + t // page_size] * page_size + t % page_size.
    Returns a list of int64 arrays, one per sequence."""
    ip = _np(page_indptr, np.int64)
    pi = _np(page_indices, np.int64)
    last = _np(last_page_len, np.int64)
    seqs = []
    for b in range(len(last)):
        pages = pi[ip[b]:ip[b + 1]]
        L = (len(pages) - 1) * page_size + last[b] if len(pages) else 0
        rows = [int(pages[t // page_size]) * page_size + t % page_size for t in range(L)]
        seqs.append(np.asarray(rows, dtype=np.int64))
    return seqs


def decode_paged(q, kv, kv_scale, page_indptr, page_indices, last_page_len, page_size: int, kv_dtype,
                 nthreads: int = 0):
    """Whole decode over a paged cache -> (out fp64 [B, 16, 512], lse fp64 [B, 16]).
    Each sequence's rows are gathered in token order (``paged_rows``) into a contiguous
    cache (with their MXFP4 block scales; the fp8 scale is per tensor) and decoded there."""
    seqs = paged_rows(page_indptr, page_indices, last_page_len, page_size)
    idx = np.concatenate(seqs) if seqs else np.zeros((0,), np.int64)
    indptr = np.zeros((len(seqs) + 1,), dtype=np.int32)
    indptr[1:] = np.cumsum([len(r) for r in seqs])
    k, s = _kv_args(kv, kv_scale, kv_dtype)
    k = np.ascontiguousarray(k[idx]) if len(idx) else np.zeros((1,) + k.shape[1:], k.dtype)
    if kv_dtype == KV_MXFP4:
        s = np.ascontiguousarray(s[idx]) if len(idx) else np.zeros((1,) + s.shape[1:], s.dtype)
    return decode(q, k, s, indptr, kv_dtype, nthreads)


def decode_paged_multi(q, qo_indptr, kv, kv_scale, page_indptr, page_indices, last_page_len, page_size: int,
                       kv_dtype, nthreads: int = 0):
    """Several query tokens per sequence -> (out fp64 [total_q, 16, 512], lse fp64 [total_q, 16]).

    Reading of the q_len > 1 form of the paged interface (qo_indptr; the pages call it only
    with one token per sequence): the q_len new tokens of sequence b are the last q_len of
    its L cached tokens, and query row qo_indptr[b] + t attends causally to the first
    L - q_len + 1 + t of them (none if that is <= 0).  Each query row is decoded on its own
    visible rows, gathered in token order by ``paged_rows``."""
    seqs = paged_rows(page_indptr, page_indices, last_page_len, page_size)
    qo = _np(qo_indptr, np.int64)
    vis = []
    for b in range(len(seqs)):
        qn = int(qo[b + 1] - qo[b])
        for t in range(qn):
            vis.append(seqs[b][:max(0, len(seqs[b]) - qn + 1 + t)])
    idx = np.concatenate(vis) if vis else np.zeros((0,), np.int64)
    indptr = np.zeros((len(vis) + 1,), dtype=np.int32)
    indptr[1:] = np.cumsum([len(r) for r in vis])
    k, s = _kv_args(kv, kv_scale, kv_dtype)
    k = np.ascontiguousarray(k[idx]) if len(idx) else np.zeros((1,) + k.shape[1:], k.dtype)
    if kv_dtype == KV_MXFP4:
        s = np.ascontiguousarray(s[idx]) if len(idx) else np.zeros((1,) + s.shape[1:], s.dtype)
    return decode(q, k, s, indptr, kv_dtype, nthreads)


def combine(o_parts, lse_parts):
    """Merge partial results of one batch row: o_parts [ns, 16, 512], lse_parts [ns, 16]."""
    lib = _load()
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    ns = o_parts.shape[0]
    out = np.zeros((NH, DV), dtype=np.float64)
    lse = np.zeros((NH,), dtype=np.float64)
    lib.mla_oracle_combine(ns, _ptr(o_parts), _ptr(lse_parts), _ptr(out), _ptr(lse))
    return out, lse


def split_range(L: int, ns: int, bn: int, s: int):
    lib = _load()
    a, b = ctypes.c_int64(0), ctypes.c_int64(0)
    lib.mla_oracle_split_range(int(L), int(ns), int(bn), int(s), ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def max_threads() -> int:
    return _load().mla_oracle_max_threads()
