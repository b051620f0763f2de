"""The no-allocation decode entry point, through the C ABI, against the entry
point that takes a caller workspace.

dcp_mla_decode_noalloc serves callers that cannot allocate device memory at
decode time (a process whose device memory another allocator reserved at
start-up, plug-in runtimes that forbid allocation after initialisation,
latency-critical paths that cannot take cudaMalloc's implicit
synchronisation): it keeps the partials in the library's built-in scratch
array. Two calls in a row, with different inputs, must each match the
workspace entry point within the tolerances of the other GPU tests. This file
is collected last, and passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import decode_context_mla_dcp_gb300 as dcp
from decode_context_mla_dcp_gb300 import build as dcp_build
from decode_context_mla_dcp_gb300.inputs import MLA_SCALE, make_mla_inputs

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 8e-3   # output tolerance of the GPU parity tests
LSE_TOL = 1e-5            # LSE tolerance of the producer tests


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _shards(kv_full, L, cp):
    B, L_max, Dk = kv_full.shape
    T = -(-L_max // cp)
    kvs, lens = [], []
    for j in range(cp):
        kv_j = np.zeros((B, T, Dk), dtype=np.uint16)
        n_j = np.zeros(B, dtype=np.int32)
        for b in range(B):
            own = np.arange(j, L[b], cp)
            kv_j[b, :own.size] = kv_full[b, own]
            n_j[b] = own.size
        kvs.append(_dev(kv_j))
        lens.append(torch.from_numpy(n_j).cuda())
    return kvs, lens, T


def _close(a, b, atol, rtol):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    same_inf = np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = np.isfinite(b)
    return same_inf and bool((np.abs(a[fin] - b[fin]) <= atol + rtol * np.abs(b[fin])).all())


def test_no_alloc_entry_point_matches_workspace_entry_point_twice():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    dcp_build.build()
    dcp.load()
    torch.cuda.set_device(0)
    cp, n_split, B, H, Dk, L_max = 4, 2, 3, 64, 576, 240
    assert dcp.dcp_mla_decode_workspace_bytes(cp, n_split, B, H) <= dcp.DCP_MLA_NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((21, 22)):
        q, kv_full = make_mla_inputs(B, H, L_max, Dk, seed=seed)
        L = np.array([L_max, 97 + call, 2], dtype=np.int32)
        kvs, lens, T = _shards(kv_full, L, cp)
        qd = _dev(q)
        ref_o = [torch.empty((B, H // cp, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
        ref_l = [torch.empty((B, H // cp), dtype=torch.float32, device="cuda") for _ in range(cp)]
        ws = torch.empty((dcp.dcp_mla_decode_workspace_bytes(cp, n_split, B, H),), dtype=torch.uint8, device="cuda")
        dcp.dcp_mla_decode(qd, kvs, lens, cp, B, H, Dk, 512, T, MLA_SCALE, True, n_split, ws, ws.numel(), ref_o,
                           ref_l)
        got_o = [torch.full((B, H // cp, 512), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
        got_l = [torch.full((B, H // cp), float("nan"), dtype=torch.float32, device="cuda") for _ in range(cp)]
        dcp.dcp_mla_decode_noalloc(qd, kvs, lens, cp, B, H, Dk, 512, T, MLA_SCALE, True, n_split, got_o, got_l)
        torch.cuda.synchronize()
        for r in range(cp):
            assert _close(got_o[r].float(), ref_o[r].float(), ATOL, RTOL), f"call {call} destination {r} output"
            assert _close(got_l[r], ref_l[r], LSE_TOL, LSE_TOL), f"call {call} destination {r} LSE"


def test_no_alloc_rejects_work_beyond_its_scratch():
    dcp.load()
    # 16 sources x 64 rows x 128 heads x (1024 + 4) bytes is about 135 MB > 32 MiB
    with pytest.raises(dcp.DcpError) as e:
        dcp.dcp_mla_decode_noalloc(1 << 20, [1 << 20] * 8, [1 << 20] * 8, 8, 64, 128, 576, 512, 100, 0.1, True, 2,
                                   [1 << 20] * 8, stream=0)
    assert e.value.status == -108
