"""GB300-native (sm_103a) LSE-weighted merge of DCP partial attention outputs.

Decode context parallelism (DCP) shards an MLA layer's KV context over cp
shards; each shard yields a partial attention output [B, H, D] and its
log-sum-exp. Destination r owns heads [r*H/cp, (r+1)*H/cp) and merges the cp
partials of those heads by LSE weight ("[DCP] Run fi_a2a on FlashInfer's fused
all-to-all + LSE reduce", "Motivation" and "Modifications"). Here all shards
are buffers on one GPU and one kernel reads them in place.

The C ABI (include/dcp_lse_reduce.h) is the product; this package is its thin
binding: ``dcp_lse_reduce`` / ``dcp_lse_reduce_ex`` take raw pointers (or
tensors) exactly like the C calls, and ``merge`` derives the sizes and strides
from torch tensors and allocates the outputs.
"""
from __future__ import annotations

from ._binding import (DCP_DTYPE_BF16, DCP_DTYPE_F16, DCP_FLAG_LSE_FIRST, DCP_FLAG_PDL, DCP_FLAG_PRELOAD,
                       DCP_LSE_REDUCE_CP_MAX, EXPORTED_SYMBOLS, DcpError, Layout, dcp_lse_reduce,
                       dcp_lse_reduce_ex, dcp_lse_reduce_strerror, dcp_lse_reduce_version, library_path, load)

__all__ = ["dcp_lse_reduce", "dcp_lse_reduce_ex", "dcp_lse_reduce_strerror", "dcp_lse_reduce_version", "merge",
           "algorithmic_bytes", "Layout", "DcpError", "load", "library_path", "EXPORTED_SYMBOLS",
           "DCP_DTYPE_BF16", "DCP_DTYPE_F16", "DCP_FLAG_PDL", "DCP_FLAG_PRELOAD", "DCP_FLAG_LSE_FIRST",
           "DCP_LSE_REDUCE_CP_MAX"]


def algorithmic_bytes(cp: int, B: int, H: int, D: int, elem: int = 2, skipped_payload_rows: int = 0) -> int:
    """HBM bytes one call must move: every source's payload and LSE read once,
    every merged output and LSE written once. ``skipped_payload_rows`` counts
    (row, head, source) payload rows with zero weight, which the kernel does
    not read."""
    return cp * B * H * D * elem + cp * B * H * 4 + B * H * D * elem + B * H * 4 - skipped_payload_rows * D * elem


def merge(srcs, lses, lse_base_e: bool, *, outs=None, lse_outs=None, flags: int = 0, stream=None,
          write_lse: bool = True, seq_lens=None, interleave: int = 1):
    """Merge cp partial outputs with the CUDA kernel.

    srcs: cp CUDA tensors [B, H, D] (bf16 or fp16; unit stride along D, other
        strides multiples of 8 elements). lses: cp fp32 tensors [B, H] or
        [B, H, 1] (any strides). Returns (outs, lse_outs): cp tensors
        [B, H/cp, D] of the sources' dtype and cp fp32 tensors [B, H/cp]
        (None entries when write_lse is False). Preallocated outs/lse_outs may
        be passed (unit stride along D). seq_lens: optional CUDA int32 [B]
        context lengths; shards owning no token of a row's context (KV
        interleaved in blocks of ``interleave`` tokens) are masked out.
    """
    import torch

    cp = len(srcs)
    if cp < 1 or len(lses) != cp:
        raise ValueError("need cp >= 1 sources and as many LSEs")
    s0 = srcs[0]
    B, H, D = s0.shape
    if H % cp:
        raise ValueError("H must be a multiple of cp")
    Hl = H // cp
    dtype = {torch.bfloat16: DCP_DTYPE_BF16, torch.float16: DCP_DTYPE_F16}.get(s0.dtype)
    if dtype is None:
        raise TypeError("sources must be bf16 or fp16")
    for s in srcs:
        if s.shape != s0.shape or s.dtype != s0.dtype or s.stride() != s0.stride() or not s.is_cuda:
            raise ValueError("sources must be CUDA tensors of one shape, dtype and stride")
        if s.stride(2) != 1:
            raise ValueError("sources need unit stride along D")
    l0 = lses[0]
    for l in lses:
        if l.dtype != torch.float32 or l.stride() != l0.stride() or l.shape[:2] != (B, H):
            raise ValueError("LSEs must be fp32 [B, H] or [B, H, 1] with one stride")
    if outs is None:
        outs = [torch.empty((B, Hl, D), dtype=s0.dtype, device=s0.device) for _ in range(cp)]
    if lse_outs is None:
        lse_outs = [torch.empty((B, Hl), dtype=torch.float32, device=s0.device) if write_lse else None
                    for _ in range(cp)]
    o0 = outs[0]
    if any(o.stride() != o0.stride() or o.stride(2) != 1 for o in outs):
        raise ValueError("outputs need one stride and unit stride along D")
    lo = next((l for l in lse_outs if l is not None), None)
    layout = Layout(src_row=s0.stride(0), src_head=s0.stride(1), lse_row=l0.stride(0), lse_head=l0.stride(1),
                    dst_row=o0.stride(0), dst_head=o0.stride(1),
                    lse_out_row=(lo.stride(0) if lo is not None else Hl))
    if seq_lens is not None and (seq_lens.dtype != torch.int32 or seq_lens.shape != (B,) or not seq_lens.is_cuda
                                 or not seq_lens.is_contiguous()):
        raise ValueError("seq_lens must be a contiguous CUDA int32 tensor of shape [B]")
    dcp_lse_reduce_ex(srcs, lses, cp, B, H, D, lse_base_e, dtype, outs,
                      [l if l is not None else 0 for l in lse_outs], layout=layout, flags=flags, stream=stream,
                      seq_lens=seq_lens, interleave=interleave)
    return outs, lse_outs
