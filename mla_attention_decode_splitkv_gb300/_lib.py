"""ctypes binding to the C ABI in include/mla_decode.h (argument marshalling only).

Every step of the decode runs in the CUDA library; this module only turns tensors into
pointers.  If the library has not been built it raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libmla_decode.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_CUDA = -3
MLA_ERR_NO_MEMORY = -4
MLA_ERR_TIMEOUT = -5

EXPORTED = (
    "mla_decode",
    "mla_decode_pick_splits",
    "mla_decode_workspace_slots",
    "mla_decode_reserve_workspace",
    "mla_decode_release_workspace",
    "mla_decode_device_status",
    "mla_decode_set_wait_limit_ns",
    "mla_decode_set_test_stall",
    "mla_decode_set_cross_rows",
    "mla_decode_profile_begin",
    "mla_decode_profile_end",
    "mla_decode_noalloc",
    "mla_decode_noalloc_status",
    "mla_decode_paged",
    "mla_decode_paged_multi",
    "mla_status_string",
    "mla_last_cuda_error",
)

_lock = threading.Lock()
_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        lib = _lib
        name = lib.mla_status_string(status).decode() if lib is not None else str(status)
        cuda = lib.mla_last_cuda_error().decode() if (lib is not None and status == MLA_ERR_CUDA) else ""
        super().__init__(f"{what}: {name}" + (f" ({cuda})" if cuda else ""))


def load(path: str = LIB_PATH):
    """Load the shared library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"MLA decode CUDA library not built ({path}); run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, c_int = ctypes.c_void_p, ctypes.c_int
        lib.mla_decode.restype = c_int
        lib.mla_decode.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, vp]
        lib.mla_decode_pick_splits.restype = c_int
        lib.mla_decode_pick_splits.argtypes = [c_int, c_int, c_int, c_int]
        lib.mla_decode_workspace_slots.restype = c_int
        lib.mla_decode_workspace_slots.argtypes = [c_int, c_int, c_int]
        lib.mla_decode_reserve_workspace.restype = c_int
        lib.mla_decode_reserve_workspace.argtypes = [c_int]
        lib.mla_decode_release_workspace.restype = c_int
        lib.mla_decode_release_workspace.argtypes = []
        lib.mla_decode_device_status.restype = c_int
        lib.mla_decode_device_status.argtypes = [c_int]
        lib.mla_decode_set_wait_limit_ns.restype = None
        lib.mla_decode_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.mla_decode_set_test_stall.restype = None
        lib.mla_decode_set_test_stall.argtypes = [c_int]
        lib.mla_decode_set_cross_rows.restype = None
        lib.mla_decode_set_cross_rows.argtypes = [c_int]
        lib.mla_decode_profile_begin.restype = c_int
        lib.mla_decode_profile_begin.argtypes = []
        lib.mla_decode_profile_end.restype = c_int
        lib.mla_decode_profile_end.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                               ctypes.POINTER(c_int)]
        lib.mla_decode_paged.restype = c_int
        lib.mla_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, c_int, vp, c_int, c_int, c_int, vp]
        lib.mla_decode_paged_multi.restype = c_int
        lib.mla_decode_paged_multi.argtypes = [vp, vp, c_int, vp, vp, vp, vp, vp, c_int, vp, c_int, c_int, c_int, vp]
        lib.mla_decode_noalloc.restype = c_int
        lib.mla_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, vp]
        lib.mla_decode_noalloc_status.restype = c_int
        lib.mla_decode_noalloc_status.argtypes = [c_int]
        lib.mla_status_string.restype = ctypes.c_char_p
        lib.mla_status_string.argtypes = [c_int]
        lib.mla_last_cuda_error.restype = ctypes.c_char_p
        lib.mla_last_cuda_error.argtypes = []
        _lib = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def mla_decode(q, kv, kv_scale, kv_indptr, out, batch: int, num_splits: int, kv_dtype: int, stream=None) -> int:
    """Raw C-ABI call with tensors (device memory); returns the mla_status code."""
    lib = load()
    return lib.mla_decode(_ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(kv_indptr), _ptr(out), int(batch),
                          int(num_splits), int(kv_dtype), _stream_handle(stream))


def decode(q, kv, kv_scale, kv_indptr, kv_dtype: int, num_splits: int = 0, out=None, stream=None):
    """out = MLA decode of q over the cache (all tensors on the GPU); raises MLAError."""
    import torch
    batch = q.shape[0]
    if out is None:
        out = torch.empty((batch, 16, 512), dtype=torch.bfloat16, device=q.device)
    rc = mla_decode(q, kv, kv_scale, kv_indptr, out, batch, num_splits, kv_dtype, stream)
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode")
    return out


def mla_decode_paged(q, kv, kv_scale, page_indptr, page_indices, last_page_len, page_size: int, out, batch: int,
                     num_splits: int, kv_dtype: int, stream=None) -> int:
    """Raw C-ABI call for a paged cache (device tensors); returns the mla_status code."""
    lib = load()
    return lib.mla_decode_paged(_ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(page_indptr), _ptr(page_indices),
                                _ptr(last_page_len), int(page_size), _ptr(out), int(batch), int(num_splits),
                                int(kv_dtype), _stream_handle(stream))


def decode_paged(q, kv, kv_scale, page_indptr, page_indices, last_page_len, page_size: int, kv_dtype: int,
                 num_splits: int = 0, out=None, stream=None):
    """out = MLA decode of q over a paged cache (all tensors on the GPU); raises MLAError."""
    import torch
    batch = q.shape[0]
    if out is None:
        out = torch.empty((batch, 16, 512), dtype=torch.bfloat16, device=q.device)
    rc = mla_decode_paged(q, kv, kv_scale, page_indptr, page_indices, last_page_len, page_size, out, batch,
                          num_splits, kv_dtype, stream)
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_paged")
    return out


def mla_decode_paged_multi(q, qo_indptr, total_q: int, kv, kv_scale, page_indptr, page_indices, last_page_len,
                           page_size: int, out, batch: int, num_splits: int, kv_dtype: int, stream=None) -> int:
    """Raw C-ABI call: several query tokens per sequence over a paged cache; returns the mla_status code."""
    lib = load()
    return lib.mla_decode_paged_multi(_ptr(q), _ptr(qo_indptr), int(total_q), _ptr(kv), _ptr(kv_scale),
                                      _ptr(page_indptr), _ptr(page_indices), _ptr(last_page_len), int(page_size),
                                      _ptr(out), int(batch), int(num_splits), int(kv_dtype), _stream_handle(stream))


def decode_paged_multi(q, qo_indptr, kv, kv_scale, page_indptr, page_indices, last_page_len, page_size: int,
                       kv_dtype: int, num_splits: int = 0, out=None, stream=None):
    """out [total_q, 16, 512] = causal multi-token MLA decode over a paged cache (GPU tensors); raises MLAError."""
    import torch
    total_q = q.shape[0]
    batch = qo_indptr.shape[0] - 1
    if out is None:
        out = torch.empty((total_q, 16, 512), dtype=torch.bfloat16, device=q.device)
    rc = mla_decode_paged_multi(q, qo_indptr, total_q, kv, kv_scale, page_indptr, page_indices, last_page_len,
                                page_size, out, batch, num_splits, kv_dtype, stream)
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_paged_multi")
    return out


def pick_splits(batch: int, kv_len_hint: int, num_sms: int, kv_dtype: int) -> int:
    rc = load().mla_decode_pick_splits(int(batch), int(kv_len_hint), int(num_sms), int(kv_dtype))
    if rc < 0:
        raise MLAError(rc, "mla_decode_pick_splits")
    return rc


def resolve_splits(num_splits, batch: int, kv_len_hint: int, num_sms: int, kv_dtype: int) -> int:
    """num_splits for mla_decode: the given value, or the library's choice when None."""
    return int(num_splits) if num_splits is not None else pick_splits(batch, kv_len_hint, num_sms, kv_dtype)


def workspace_slots(batch: int, num_splits: int, num_sms: int) -> int:
    rc = load().mla_decode_workspace_slots(int(batch), int(num_splits), int(num_sms))
    if rc < 0:
        raise MLAError(rc, "mla_decode_workspace_slots")
    return rc


def reserve_workspace(slots: int) -> None:
    rc = load().mla_decode_reserve_workspace(int(slots))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_reserve_workspace")


def release_workspace() -> None:
    rc = load().mla_decode_release_workspace()
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_release_workspace")


def device_status(clear: bool = True) -> int:
    return load().mla_decode_device_status(1 if clear else 0)


def set_wait_limit_ns(ns: int) -> None:
    load().mla_decode_set_wait_limit_ns(int(ns))


def set_test_stall(on: bool) -> None:
    """Test hook: make every mla_decode call's pipeline wait run past its limit."""
    load().mla_decode_set_test_stall(1 if on else 0)


def set_cross_rows(rows: int) -> None:
    """Test hook: the balanced mode's crossing cost in cache rows (< 0: the default)."""
    load().mla_decode_set_cross_rows(int(rows))


def profile_begin() -> None:
    load().mla_decode_profile_begin()


def profile_end():
    """-> (summed split-kernel ms, summed call ms, number of calls)."""
    a, b, n = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_int(0)
    rc = load().mla_decode_profile_end(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_profile_end")
    return a.value, b.value, n.value


def mla_decode_noalloc(q, kv, kv_scale, kv_indptr, out, batch: int, num_splits: int, kv_dtype: int,
                       stream=None) -> int:
    """Raw C-ABI call of the allocation-free variant (device tensors); returns the status."""
    lib = load()
    return lib.mla_decode_noalloc(_ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(kv_indptr), _ptr(out), int(batch),
                                  int(num_splits), int(kv_dtype), _stream_handle(stream))


def noalloc_status(clear: bool = True) -> int:
    """Status of the most recent mla_decode_noalloc call (MLA_OK or MLA_ERR_TIMEOUT)."""
    return load().mla_decode_noalloc_status(1 if clear else 0)
