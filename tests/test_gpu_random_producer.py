"""Seeded random cases of the producer (split-KV MLA decode attention over
one shard) against the fp64 oracle attention: heads 16..192, Dk 512 or 576,
cache lengths 1..900, 1..8 splits, per-row token counts from 0 to past the
cache (clamped), base 2 or e, PDL and the prefetch flag, each kernel forced
and the default choice. Cache rows at and past a row's token count hold NaN
and must not reach any output."""
import numpy as np
import pytest
import torch

import decode_context_mla_dcp_gb300 as dcp
from decode_context_mla_dcp_gb300 import build as dcp_build
from decode_context_mla_dcp_gb300.inputs import MLA_SCALE, make_mla_inputs
from tests.test_gpu_mla import check_lse, check_out, dev_bf16, oracle_partials

pytestmark = pytest.mark.gpu

KERNEL_FLAGS = [0, dcp.DCP_MLA_FLAG_TCGEN05, dcp.DCP_MLA_FLAG_MMA_SYNC]


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    dcp_build.build()
    dcp.load()
    torch.cuda.set_device(0)
    yield


@pytest.mark.parametrize("case", range(24))
def test_random_producer_calls_match_the_oracle(oracle_mod, case):
    rng = np.random.default_rng([77, case])
    H = 16 * int(rng.integers(1, 13))
    Dk = int(rng.choice([512, 576]))
    T = int(rng.integers(1, 901))
    B = int(rng.integers(1, 6))
    n_split = int(rng.integers(1, 9))
    base_e = bool(rng.integers(0, 2))
    flags = KERNEL_FLAGS[case % 3] | int(rng.choice([0, dcp.DCP_FLAG_PDL, dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH]))
    lens = rng.integers(0, T + 6, size=B).astype(np.int32)
    lens[0] = T
    if B > 1:
        lens[1] = 0
    q, kv = make_mla_inputs(B, H, T, Dk, seed=1000 + case)
    for b in range(B):
        kv[b, min(int(lens[b]), T):] = 0x7FC0  # NaN rows: not this row's tokens
    outs, lses = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), torch.from_numpy(lens).cuda(), MLA_SCALE,
                                        lse_base_e=base_e, n_split=n_split, flags=flags)
    torch.cuda.synchronize()
    what = f"H={H} Dk={Dk} T={T} B={B} n_split={n_split} base_e={base_e} flags={flags} lens={lens.tolist()}"
    ref_o, ref_l = oracle_partials(q, kv, np.minimum(lens, T), n_split, MLA_SCALE, base_e)
    for s in range(n_split):
        check_out(outs[s], ref_o[s], f"split {s}, {what}")
        check_lse(lses[s], ref_l[s], f"split {s}, {what}")


@pytest.mark.parametrize("case", range(16))
def test_random_fused_decodes_match_full_attention(oracle_mod, case):
    """dcp_mla_decode on random shard counts, splits, heads and row lengths
    (the context interleaved token by token over the shards), the two-launch
    default and the one-kernel flag, against fp64 attention over each row's
    whole context."""
    from oracle.attention import attention
    from tests.test_gpu_mla import _interleaved_shards, widen

    rng = np.random.default_rng([88, case])
    cp = int(rng.choice([1, 2, 4, 8]))
    n_split = int(rng.integers(1, 16 // cp + 1))
    Hs = 16 * int(rng.integers(1, 3))                 # heads per (shard, split) block of the merge
    H = Hs * cp * n_split if Hs * cp * n_split <= 192 else 16 * cp * n_split
    Dk = int(rng.choice([512, 576]))
    B = int(rng.integers(1, 5))
    L_max = int(rng.integers(1, 700))
    L = rng.integers(0, L_max + 1, size=B).astype(np.int32)
    L[0] = L_max
    flags = int(rng.choice([0, dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH])) | \
        (dcp.DCP_MLA_FLAG_ONE_KERNEL if case % 2 else 0)
    q, kv_full = make_mla_inputs(B, H, L_max, Dk, seed=2000 + case)
    kvs, lens = _interleaved_shards(kv_full, L, cp)
    outs, louts = dcp.mla_decode_dcp(dev_bf16(q), kvs, lens, MLA_SCALE, n_split=n_split, flags=flags)
    torch.cuda.synchronize()
    what = f"cp={cp} n_split={n_split} H={H} Dk={Dk} B={B} L={L.tolist()} flags={flags}"
    Hl = H // cp
    for b in range(B):
        o_ref, l_ref = attention(widen(q[b:b + 1]), widen(kv_full[b, :L[b]]), MLA_SCALE, dv=512)
        for r in range(cp):
            check_out(outs[r][b:b + 1], o_ref[:, r * Hl:(r + 1) * Hl], f"row {b} dest {r}, {what}",
                      kind="fused decode")
            check_lse(louts[r][b:b + 1], l_ref[:, r * Hl:(r + 1) * Hl], f"row {b} dest {r}, {what}",
                      kind="fused decode")
