"""CPU oracle for the DCP LSE-weighted merge.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product path (the CUDA
library and its binding) never imports this package, and this package never
imports the product.

* ``merge`` wraps ``dcp_merge_oracle.c``: a plain fp64 loop nest over
  (destination, row, local head, feature) that states the merge exactly as the
  pages describe it (sources cited in that file).
* ``attention`` holds a brute-force fp64 softmax attention used to produce
  split-context partials for the tiny exactness check and to pin the merge
  against full-context attention.

Parity of ``merge`` is pinned by closed forms (tests/test_oracle_pins.py and
tests/golden/): the identity at cp = 1, the exact mean at equal LSEs, zero
weight for -inf shards, base-2/base-e agreement, shift invariance,
associativity of nested merges, one-hot head routing, and equality with
brute-force full-context attention.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = ["merge", "half_bits_to_double", "build", "library_path", "open_library"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dcp_merge_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libdcp_merge_oracle.so")

_BF16, _F16, _F64 = 0, 1, 2
_LSE_F32, _LSE_F64 = 0, 1

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math, no FMA contraction)."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        os.makedirs(_BUILD_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def open_library(path: str):
    """Open a compiled oracle at ``path`` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.oracle_dcp_merge.argtypes = [
        ctypes.c_int, ctypes.POINTER(vp), ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int, ctypes.POINTER(vp), ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_int,
        ctypes.POINTER(vp), ctypes.POINTER(vp)]
    lib.oracle_dcp_merge.restype = ctypes.c_int
    lib.oracle_half_bits_to_double.argtypes = [ctypes.c_int, ctypes.c_uint16]
    lib.oracle_half_bits_to_double.restype = ctypes.c_double
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = open_library(_LIB_PATH)
    return _lib


def merge(srcs, lses, lse_base_e: bool, *, dtype: str = "bf16", H: int | None = None,
          D: int | None = None, src_strides: tuple[int, int] | None = None,
          lse_strides: tuple[int, int] | None = None, seq_lens=None, interleave: int = 1):
    """Merge cp partial outputs into cp destinations, in fp64.

    srcs: cp arrays. For dtype 'bf16'/'f16' they hold raw 16-bit patterns
        (np.uint16); for dtype 'f64' they are float64. Each is indexed as
        flat[b*src_row + h*src_head + d]; the default strides are those of a
        contiguous [B, H, D] array.
    lses: cp float32 (or float64) arrays indexed flat[b*lse_row + h*lse_head];
        the default is contiguous [B, H] (FlashMLA's [B, H, 1] is the same).
    seq_lens: optional [B] context lengths; with the KV interleaved over the
        shards in blocks of ``interleave`` tokens, a shard that owns no token
        of a row's context is empty for that row (LSE ignored, weight 0).
    Returns (outs, lse_outs): cp arrays of shape [B, H/cp, D] and [B, H/cp],
    float64.
    """
    cp = len(srcs)
    if cp != len(lses) or cp < 1:
        raise ValueError("srcs and lses must both have cp >= 1 entries")
    s0 = np.asarray(srcs[0])
    if src_strides is None:
        if s0.ndim != 3:
            raise ValueError("default strides need [B, H, D] sources")
        B, Hs, D = s0.shape
        src_strides = (Hs * D, D)
        H = Hs if H is None else H
    else:
        # explicit strides: sources are [B, ...] backing arrays; H and D given
        # or taken from a [B, H, D]-shaped array
        if s0.ndim < 2:
            raise ValueError("explicit strides need [B, ...]-shaped sources")
        B = s0.shape[0]
        if H is None or D is None:
            if s0.ndim != 3:
                raise ValueError("pass H and D for non-[B, H, D] backing arrays")
            H = s0.shape[1] if H is None else H
            D = s0.shape[2] if D is None else D
    if lse_strides is None:
        lse_strides = (H, 1)
    code = {"bf16": _BF16, "f16": _F16, "f64": _F64}[dtype]
    want = np.float64 if code == _F64 else np.uint16
    if any(np.asarray(s).dtype != want for s in srcs):
        raise TypeError(f"dtype {dtype!r} needs {want.__name__} source arrays")
    src_arrays = [np.ascontiguousarray(s) for s in srcs]
    lse_dt = np.asarray(lses[0]).dtype
    if lse_dt not in (np.float32, np.float64):
        raise TypeError("LSEs must be float32 or float64")
    lse_arrays = [np.ascontiguousarray(l, dtype=lse_dt) for l in lses]
    lse_code = _LSE_F32 if lse_dt == np.float32 else _LSE_F64
    if H % cp != 0:
        raise ValueError("H must be divisible by cp")
    Hl = H // cp
    outs = [np.empty((B, Hl, D), dtype=np.float64) for _ in range(cp)]
    lse_outs = [np.empty((B, Hl), dtype=np.float64) for _ in range(cp)]

    sl = None
    if seq_lens is not None:
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        if sl.shape != (B,):
            raise ValueError("seq_lens must have one entry per row")
    vp = ctypes.c_void_p
    arr = vp * cp
    lib = _load()
    rc = lib.oracle_dcp_merge(
        code, arr(*[a.ctypes.data for a in src_arrays]), src_strides[0], src_strides[1],
        lse_code, arr(*[a.ctypes.data for a in lse_arrays]), lse_strides[0], lse_strides[1],
        cp, B, H, D, 1 if lse_base_e else 0,
        sl.ctypes.data if sl is not None else None, int(interleave),
        arr(*[o.ctypes.data for o in outs]), arr(*[o.ctypes.data for o in lse_outs]))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return outs, lse_outs


def half_bits_to_double(dtype: str, bits: int) -> float:
    """The oracle's widening of one bf16/f16 bit pattern (exposed for pinning)."""
    return _load().oracle_half_bits_to_double({"bf16": _BF16, "f16": _F16}[dtype], bits)
