"""ctypes binding of the C ABI in include/dcp_lse_reduce.h.

Argument marshalling only: every step of the merge runs in the sm_103a kernel.
Pointers may be given as integers or as torch tensors (their data_ptr()); a
stream may be None (torch's current stream), an integer cudaStream_t or a
torch.cuda.Stream. A nonzero status raises DcpError carrying the library's
message. There is no fallback: if the library is not built, the first call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

DCP_LSE_REDUCE_CP_MAX = 16
DCP_DTYPE_BF16 = 0
DCP_DTYPE_F16 = 1
DCP_FLAG_PDL = 1
DCP_FLAG_PRELOAD = 2
DCP_FLAG_LSE_FIRST = 4
DCP_FLAG_PREFETCH = 8

EXPORTED_SYMBOLS = ("dcp_lse_reduce", "dcp_lse_reduce_ex", "dcp_lse_reduce_strerror", "dcp_lse_reduce_version",
                    "dcp_mla_decode_partial", "dcp_mla_decode_smem_bytes", "dcp_mla_decode_workspace_bytes",
                    "dcp_mla_decode", "dcp_mla_decode_noalloc", "dcp_mla_decode_kernel", "dcp_mla_decode_pick_split")
DCP_MLA_NOALLOC_SCRATCH_BYTES = 32 << 20
DCP_MLA_SPLIT_MAX = 16
DCP_MLA_FLAG_MMA_SYNC = 2
DCP_MLA_FLAG_TCGEN05 = 4
DCP_MLA_FLAG_ONE_KERNEL = 16
DCP_MLA_FLAG_TEST_STALL = 32
DCP_MLA_KERNEL_TCGEN05 = 1
DCP_MLA_KERNEL_MMA_SYNC = 2
DCP_LSE_REDUCE_INTERLEAVE_MAX = 1 << 24


class DcpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dcp_lse_reduce failed ({status}): {message}")
        self.status = status


class Layout(ctypes.Structure):
    """Strides in elements; mirrors dcp_lse_reduce_layout."""
    _fields_ = [("src_row", ctypes.c_int64), ("src_head", ctypes.c_int64),
                ("lse_row", ctypes.c_int64), ("lse_head", ctypes.c_int64),
                ("dst_row", ctypes.c_int64), ("dst_head", ctypes.c_int64),
                ("lse_out_row", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Open the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(
                f"the sm_103a library is not built ({p} missing): run "
                "`python -m decode_context_mla_dcp_gb300.build` or __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.dcp_lse_reduce.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i64, ci, i64, ci, ci, ci,
                                       ctypes.POINTER(vp), ctypes.POINTER(vp), vp]
        lib.dcp_lse_reduce.restype = ci
        lib.dcp_lse_reduce_ex.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ci, i64, ci, ci, ci, ci,
                                          ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(Layout),
                                          vp, ci, ctypes.c_uint, vp]
        lib.dcp_lse_reduce_ex.restype = ci
        lib.dcp_lse_reduce_strerror.argtypes = [ci]
        lib.dcp_lse_reduce_strerror.restype = ctypes.c_char_p
        lib.dcp_lse_reduce_version.argtypes = []
        lib.dcp_lse_reduce_version.restype = ci
        lib.dcp_mla_decode_partial.argtypes = [vp, vp, vp, i64, ci, ci, ci, i64, ctypes.c_float, ci, ci,
                                               ctypes.POINTER(vp), ctypes.POINTER(vp), vp, ctypes.c_uint, vp]
        lib.dcp_mla_decode_partial.restype = ci
        lib.dcp_mla_decode_smem_bytes.argtypes = [ci, ci]
        lib.dcp_mla_decode_smem_bytes.restype = ci
        lib.dcp_mla_decode_kernel.argtypes = [ci, i64, ci, ctypes.c_uint]
        lib.dcp_mla_decode_kernel.restype = ci
        lib.dcp_mla_decode_pick_split.argtypes = [ci, i64, ci, i64, ci]
        lib.dcp_mla_decode_pick_split.restype = ci
        lib.dcp_mla_decode_workspace_bytes.argtypes = [ci, ci, i64, ci, ci]
        lib.dcp_mla_decode_workspace_bytes.restype = i64
        lib.dcp_mla_decode.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ci, i64, ci, ci, ci, i64,
                                       ctypes.c_float, ci, ci, vp, i64, ctypes.POINTER(vp), ctypes.POINTER(vp), vp,
                                       ctypes.c_uint, vp]
        lib.dcp_mla_decode.restype = ci
        lib.dcp_mla_decode_noalloc.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ci, i64, ci, ci, ci, i64,
                                               ctypes.c_float, ci, ci, ctypes.POINTER(vp), ctypes.POINTER(vp), vp,
                                               ctypes.c_uint, vp]
        lib.dcp_mla_decode_noalloc.restype = ci
        if path is None:
            _lib = lib
        return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(xs, n: int, allow_none: bool = False):
    if xs is None:
        if allow_none:
            return None
        raise ValueError("pointer array is required")
    vals = [_ptr(x) for x in xs]
    if len(vals) < n:
        raise ValueError(f"need {n} pointers, got {len(vals)}")
    return (ctypes.c_void_p * len(vals))(*vals)


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int) -> None:
    if status != 0:
        raise DcpError(status, dcp_lse_reduce_strerror(status))


def dcp_lse_reduce(src_ptrs, lse_ptrs, lse_stride: int, cp: int, B: int, H: int, D: int, lse_base_e: bool,
                   dst_ptrs, lse_out_ptrs=None, stream=None) -> None:
    """The merge over contiguous [B, H, D] bf16 buffers (see the C header)."""
    lib = load()
    _check(lib.dcp_lse_reduce(_ptr_array(src_ptrs, cp), _ptr_array(lse_ptrs, cp), int(lse_stride), int(cp),
                              int(B), int(H), int(D), 1 if lse_base_e else 0, _ptr_array(dst_ptrs, cp),
                              _ptr_array(lse_out_ptrs, cp, allow_none=True), _stream(stream)))


def dcp_lse_reduce_ex(src_ptrs, lse_ptrs, cp: int, B: int, H: int, D: int, lse_base_e: bool,
                      dtype: int, dst_ptrs, lse_out_ptrs=None, layout: Layout | dict | None = None,
                      flags: int = 0, stream=None, seq_lens=None, interleave: int = 1) -> None:
    """The merge with explicit strides, dtype, empty-shard masking from
    per-row context lengths (``seq_lens``: device int32 [B], KV interleaved
    in blocks of ``interleave`` tokens) and launch flags (see the C header)."""
    lib = load()
    if isinstance(layout, dict):
        layout = Layout(**layout)
    _check(lib.dcp_lse_reduce_ex(_ptr_array(src_ptrs, cp), _ptr_array(lse_ptrs, cp), int(cp), int(B), int(H),
                                 int(D), 1 if lse_base_e else 0, int(dtype), _ptr_array(dst_ptrs, cp),
                                 _ptr_array(lse_out_ptrs, cp, allow_none=True),
                                 ctypes.byref(layout) if layout is not None else None, _ptr(seq_lens),
                                 int(interleave), int(flags), _stream(stream)))


def dcp_lse_reduce_strerror(status: int) -> str:
    return load().dcp_lse_reduce_strerror(int(status)).decode()


def dcp_mla_decode_partial(q, kv, kv_len, B: int, H: int, Dk: int, Dv: int, T: int, scale: float,
                           lse_base_e: bool, n_split: int, out_ptrs, lse_ptrs, status=None, flags: int = 0,
                           stream=None) -> None:
    """Split-KV MLA decode attention over one shard (see include/dcp_mla_decode.h)."""
    lib = load()
    _check(lib.dcp_mla_decode_partial(_ptr(q), _ptr(kv), _ptr(kv_len), int(B), int(H), int(Dk), int(Dv), int(T),
                                      float(scale), 1 if lse_base_e else 0, int(n_split),
                                      _ptr_array(out_ptrs, n_split), _ptr_array(lse_ptrs, n_split), _ptr(status),
                                      int(flags), _stream(stream)))


def dcp_mla_decode_smem_bytes(Dk: int, H: int) -> int:
    return int(load().dcp_mla_decode_smem_bytes(int(Dk), int(H)))


def dcp_mla_decode_pick_split(cp: int, B: int, H: int, T: int, num_sms: int) -> int:
    """A one-wave split count for cp shards (see the C header; host only)."""
    n = int(load().dcp_mla_decode_pick_split(int(cp), int(B), int(H), int(T), int(num_sms)))
    if n < 0:
        _check(n)
    return n


def dcp_mla_decode_kernel(H: int, T: int, n_split: int, flags: int = 0) -> int:
    """DCP_MLA_KERNEL_TCGEN05 or DCP_MLA_KERNEL_MMA_SYNC: the producer kernel
    these arguments select (host only; raises DcpError for invalid ones)."""
    k = int(load().dcp_mla_decode_kernel(int(H), int(T), int(n_split), int(flags)))
    if k < 0:
        _check(k)
    return k


def dcp_mla_decode_workspace_bytes(cp: int, n_split: int, B: int, H: int, Dv: int = 512) -> int:
    return int(load().dcp_mla_decode_workspace_bytes(int(cp), int(n_split), int(B), int(H), int(Dv)))


def dcp_mla_decode(q, kv_ptrs, kv_len_ptrs, cp: int, B: int, H: int, Dk: int, Dv: int, T: int, scale: float,
                   lse_base_e: bool, n_split: int, workspace, workspace_bytes: int, dst_ptrs, lse_out_ptrs=None,
                   status=None, flags: int = 0, stream=None) -> None:
    """Producer over cp shards + merge into cp destinations (see include/dcp_mla_decode.h)."""
    lib = load()
    _check(lib.dcp_mla_decode(_ptr(q), _ptr_array(kv_ptrs, cp), _ptr_array(kv_len_ptrs, cp), int(cp), int(B),
                              int(H), int(Dk), int(Dv), int(T), float(scale), 1 if lse_base_e else 0, int(n_split),
                              _ptr(workspace), int(workspace_bytes), _ptr_array(dst_ptrs, cp),
                              _ptr_array(lse_out_ptrs, cp, allow_none=True), _ptr(status), int(flags),
                              _stream(stream)))


def dcp_lse_reduce_version() -> int:
    return int(load().dcp_lse_reduce_version())


def dcp_mla_decode_noalloc(q, kv_ptrs, kv_len_ptrs, cp: int, B: int, H: int, Dk: int, Dv: int, T: int,
                           scale: float, lse_base_e: bool, n_split: int, dst_ptrs, lse_out_ptrs=None, status=None,
                           flags: int = 0, stream=None) -> None:
    """dcp_mla_decode with the partials in the library's built-in scratch
    array instead of a caller workspace, for callers that cannot allocate
    device memory when they decode (see include/dcp_mla_decode.h: the limit,
    the first-call set-up, and why overlapping calls race)."""
    lib = load()
    _check(lib.dcp_mla_decode_noalloc(_ptr(q), _ptr_array(kv_ptrs, cp), _ptr_array(kv_len_ptrs, cp), int(cp), int(B),
                                      int(H), int(Dk), int(Dv), int(T), float(scale), 1 if lse_base_e else 0,
                                      int(n_split), _ptr_array(dst_ptrs, cp),
                                      _ptr_array(lse_out_ptrs, cp, allow_none=True), _ptr(status), int(flags),
                                      _stream(stream)))
