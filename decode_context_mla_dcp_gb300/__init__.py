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
                       DCP_FLAG_PREFETCH,
                       DCP_LSE_REDUCE_CP_MAX, DCP_MLA_FLAG_MMA_SYNC, DCP_MLA_FLAG_TCGEN05, DCP_MLA_FLAG_ONE_KERNEL,
                       DCP_MLA_FLAG_TEST_STALL,
                       DCP_MLA_SPLIT_MAX,
                       DCP_MLA_KERNEL_MMA_SYNC, DCP_MLA_KERNEL_TCGEN05, dcp_mla_decode_kernel,
                       dcp_mla_decode_pick_split,
                       EXPORTED_SYMBOLS, DcpError,
                       Layout,
                       dcp_lse_reduce, dcp_lse_reduce_ex, dcp_lse_reduce_strerror, dcp_lse_reduce_version,
                       DCP_MLA_NOALLOC_SCRATCH_BYTES, dcp_mla_decode, dcp_mla_decode_noalloc,
                       dcp_mla_decode_partial, dcp_mla_decode_smem_bytes,
                       dcp_mla_decode_workspace_bytes, library_path, load)

__all__ = ["dcp_lse_reduce", "dcp_lse_reduce_ex", "dcp_lse_reduce_strerror", "dcp_lse_reduce_version", "merge",
           "dcp_mla_decode_partial", "dcp_mla_decode_smem_bytes", "mla_decode_partial", "DCP_MLA_SPLIT_MAX",
           "dcp_mla_decode", "dcp_mla_decode_workspace_bytes", "mla_decode_dcp", "dcp_mla_decode_noalloc",
           "DCP_MLA_NOALLOC_SCRATCH_BYTES", "DCP_MLA_FLAG_MMA_SYNC", "DCP_MLA_FLAG_TCGEN05",
           "DCP_MLA_FLAG_ONE_KERNEL", "DCP_MLA_FLAG_TEST_STALL",
           "algorithmic_bytes", "Layout", "DcpError", "load", "library_path", "EXPORTED_SYMBOLS",
           "DCP_DTYPE_BF16", "DCP_DTYPE_F16", "DCP_FLAG_PDL", "DCP_FLAG_PRELOAD", "DCP_FLAG_LSE_FIRST",
           "DCP_FLAG_PREFETCH",
           "DCP_LSE_REDUCE_CP_MAX", "dcp_mla_decode_kernel", "DCP_MLA_KERNEL_TCGEN05", "DCP_MLA_KERNEL_MMA_SYNC",
           "dcp_mla_decode_pick_split"]


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


def _num_sms(device) -> int:
    import torch
    return int(torch.cuda.get_device_properties(device).multi_processor_count)


def mla_decode_partial(q, kv, kv_len, scale: float, *, lse_base_e: bool = True, n_split: int | None = 1,
                       dv: int = 512, outs=None, lses=None, status=None, flags: int = 0, stream=None):
    """Split-KV MLA decode attention over one shard with the CUDA kernel.

    q: CUDA bf16 [B, H, Dk]; kv: CUDA bf16 [B, T, Dk] (row b's shard-local
    tokens); kv_len: CUDA int32 [B]. Returns (outs, lses): n_split bf16
    [B, H, dv] partial outputs and n_split fp32 [B, H] LSEs, one per contiguous
    token range of each row. n_split=None picks a one-wave split count
    (dcp_mla_decode_pick_split).
    """
    import torch

    B, H, Dk = q.shape
    T = kv.shape[1]
    if n_split is None:
        n_split = dcp_mla_decode_pick_split(1, B, H, T, _num_sms(q.device))
    if q.dtype != torch.bfloat16 or kv.dtype != torch.bfloat16 or not (q.is_contiguous() and kv.is_contiguous()):
        raise ValueError("q and kv must be contiguous bf16 CUDA tensors")
    if kv.shape[0] != B or kv.shape[2] != Dk or kv_len.dtype != torch.int32 or kv_len.shape != (B,):
        raise ValueError("kv must be [B, T, Dk] and kv_len int32 [B]")
    if outs is None:
        outs = [torch.empty((B, H, dv), dtype=torch.bfloat16, device=q.device) for _ in range(n_split)]
    if lses is None:
        lses = [torch.empty((B, H), dtype=torch.float32, device=q.device) for _ in range(n_split)]
    dcp_mla_decode_partial(q, kv, kv_len, B, H, Dk, dv, T, scale, lse_base_e, n_split, outs, lses, status=status,
                           flags=flags, stream=stream)
    return outs, lses


def mla_decode_dcp(q, kvs, kv_lens, scale: float, *, n_split: int | None = 1, lse_base_e: bool = True,
                   dv: int = 512, workspace=None, outs=None, lse_outs=None, status=None, flags: int = 0,
                   stream=None):
    """DCP decode attention on one GPU: the producer over each shard in
    ``kvs`` (bf16 [B, T, Dk] each, token counts ``kv_lens`` int32 [B] each),
    then the merge into cp destinations. Returns (outs, lse_outs): cp bf16
    [B, H/cp, dv] and cp fp32 [B, H/cp]. The workspace (a uint8 CUDA tensor of
    at least dcp_mla_decode_workspace_bytes bytes) is allocated with torch
    when not given. n_split=None picks a one-wave split count
    (dcp_mla_decode_pick_split)."""
    import torch

    cp = len(kvs)
    B, H, Dk = q.shape
    T = kvs[0].shape[1]
    if n_split is None:
        n_split = dcp_mla_decode_pick_split(cp, B, H, T, _num_sms(q.device))
    need = dcp_mla_decode_workspace_bytes(cp, n_split, B, H, dv)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
    if outs is None:
        outs = [torch.empty((B, H // cp, dv), dtype=torch.bfloat16, device=q.device) for _ in range(cp)]
    if lse_outs is None:
        lse_outs = [torch.empty((B, H // cp), dtype=torch.float32, device=q.device) for _ in range(cp)]
    dcp_mla_decode(q, kvs, kv_lens, cp, B, H, Dk, dv, T, scale, lse_base_e, n_split, workspace,
                   workspace.numel() * workspace.element_size(), outs, lse_outs, status=status, flags=flags,
                   stream=stream)
    return outs, lse_outs
