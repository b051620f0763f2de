"""GPU parity of the DCP producer (split-KV MLA decode attention per shard)
against the fp64 oracle attention, and of producer + merge against attention
over the whole context.

Tolerances: partial outputs |gpu - ref| <= 1e-2 + 8e-3*|ref| (bf16
probabilities and bf16 output rounding dominate: about 2^-9 relative each);
LSEs |gpu - ref| <= 1e-5 * max(|ref|, 1), the merge's LSE tolerance (fp32
scores accumulated over Dk <= 576 bf16 products, hardware exp2 at ~2 ulp,
fp32 sums over the tokens; the worst error these tests record is printed at
the end of the run).
"""
import math

import numpy as np
import pytest
import torch

import decode_context_mla_dcp_gb300 as dcp
from decode_context_mla_dcp_gb300 import build as dcp_build
from decode_context_mla_dcp_gb300.inputs import MLA_SCALE, bf16_bits, make_mla_inputs, tiny_qkv
from tests.conftest import record_error

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 8e-3
LSE_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    dcp_build.build()
    dcp.load()
    torch.cuda.set_device(0)
    yield


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def widen(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_out(got, ref, what, kind="producer"):
    got = got.float().double().cpu().numpy() if torch.is_tensor(got) else got
    assert not np.isnan(got).any(), what
    err = np.abs(got - ref)
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"{what}: max err {err.max():.3g}"
    record_error(f"{kind} output |gpu - oracle|", float(err.max()))
    return float(err.max())


def check_lse(got, ref, what, kind="producer"):
    got = got.double().cpu().numpy() if torch.is_tensor(got) else got
    ninf = ref == -np.inf
    assert np.array_equal(got == -np.inf, ninf), f"{what}: -inf pattern"
    err = np.abs(got[~ninf] - ref[~ninf])
    rel = err / np.maximum(np.abs(ref[~ninf]), 1)
    assert (rel <= LSE_TOL).all(), f"{what}: LSE max err {err.max() if err.size else 0:.3g}"
    if rel.size:
        record_error(f"{kind} LSE |gpu - oracle| / max(|oracle|, 1)", float(rel.max()))
    return float(err.max()) if err.size else 0.0


def oracle_partials(q_bits, kv_bits, lens, n_split, scale, base_e, dv=512):
    """Oracle per (row, split): attention over the split's token range."""
    from oracle.attention import attention
    q = widen(q_bits)
    kv = widen(kv_bits)
    B, H, _ = q.shape
    outs = [np.zeros((B, H, dv)) for _ in range(n_split)]
    lses = [np.full((B, H), -np.inf) for _ in range(n_split)]
    for b in range(B):
        L = int(lens[b])
        chunk = -(-L // n_split)
        for s in range(n_split):
            t0, t1 = s * chunk, min(L, (s + 1) * chunk)
            if t1 > t0:
                o, l = attention(q[b:b + 1], kv[b, t0:t1], scale, base_e, dv)
                outs[s][b], lses[s][b] = o[0], l[0]
    return outs, lses


KERNELS = [dcp.DCP_MLA_FLAG_TCGEN05, dcp.DCP_MLA_FLAG_MMA_SYNC]


@pytest.mark.parametrize("kflags", KERNELS)
@pytest.mark.parametrize("H,Dk,T,n_split", [(16, 576, 100, 1), (64, 576, 257, 3), (128, 576, 96, 2),
                                            (32, 512, 64, 1), (16, 512, 33, 16), (64, 576, 700, 2),
                                            (64, 512, 300, 1), (96, 576, 400, 1), (192, 576, 260, 1)])
@pytest.mark.parametrize("base_e", [True, False])
def test_partials_match_oracle(oracle_mod, H, Dk, T, n_split, base_e, kflags):
    B = 4
    q, kv = make_mla_inputs(B, H, T, Dk, seed=H + T)
    lens = np.array([T, 1, 0, T - 5 if T > 5 else T], dtype=np.int32)
    outs, lses = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), torch.from_numpy(lens).cuda(), MLA_SCALE,
                                        lse_base_e=base_e, n_split=n_split, flags=kflags)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_partials(q, kv, lens, n_split, MLA_SCALE, base_e)
    for s in range(n_split):
        check_out(outs[s], ref_o[s], f"split {s}")
        check_lse(lses[s], ref_l[s], f"split {s}")


@pytest.mark.parametrize("kflags", KERNELS)
@pytest.mark.parametrize("H,T,n_split", [(64, 700, 2), (128, 300, 1), (32, 520, 2), (16, 200, 3), (64, 1000, 5)])
def test_cache_rows_past_kv_len_may_hold_nan(oracle_mod, H, T, n_split, kflags):
    """Cache rows at and past a row's kv_len are not the row's tokens and may
    hold anything: filled with NaN here, they must not reach any output
    (among them the tiles that run past a split's end, and, for the last row,
    past the cache)."""
    B, Dk = 5, 576
    q, kv = make_mla_inputs(B, H, T, Dk, seed=3 * H + T)
    lens = np.array([T, T - 1, T // 2 + 3, 130, 0], dtype=np.int32)
    for b in range(B):
        kv[b, lens[b]:] = 0x7FC0
    outs, lses = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), torch.from_numpy(lens).cuda(), MLA_SCALE,
                                        n_split=n_split, flags=kflags)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_partials(q, kv, lens, n_split, MLA_SCALE, True)
    for s_ in range(n_split):
        check_out(outs[s_], ref_o[s_], f"split {s_}")
        check_lse(lses[s_], ref_l[s_], f"split {s_}")


def test_tiny_exactness_producer_then_merge(oracle_mod):
    """The tiny exactness check end to end on the GPU: two shards of 32
    tokens each, producer per shard, merge; equals attention over all 64."""
    from oracle.attention import attention
    q32, kv32 = tiny_qkv(0)
    q = bf16_bits(q32)                                   # [3, 16, 512]
    kv = np.broadcast_to(bf16_bits(kv32), (3, 64, 512)).copy()
    scale = 1 / math.sqrt(512)
    parts, part_l = [], []
    for j in range(2):
        o, l = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv[:, 32 * j:32 * j + 32].copy()),
                                      torch.full((3,), 32, dtype=torch.int32, device="cuda"), scale)
        parts.append(o[0])
        part_l.append(l[0])
    outs, louts = dcp.merge(parts, part_l, True)
    torch.cuda.synchronize()
    o_full, l_full = attention(widen(q), widen(kv[0]), scale)
    check_out(torch.cat(outs, 1), o_full, "tiny merged output", kind="producer+merge")
    check_lse(torch.cat(louts, 1), l_full, "tiny merged LSE", kind="producer+merge")


@pytest.mark.parametrize("cp,n_split,H", [(4, 2, 64), (8, 2, 128), (2, 8, 16)])
def test_dcp_composition_equals_full_attention(oracle_mod, cp, n_split, H):
    """Interleaved context shards (token t on shard t % cp), producer per
    shard with in-shard splits, one merge over all cp*n_split partials into a
    single [B, H, 512] output: attention over every row's whole context."""
    from oracle.attention import attention
    B, L_max, Dk = 3, 300, 576
    q, kv_full = make_mla_inputs(B, H, L_max, Dk, seed=cp * 10 + n_split)
    L = np.array([L_max, 37, cp - 1], dtype=np.int32)  # the last row leaves one shard empty
    parts, part_l = [], []
    for j in range(cp):
        T_j = -(-L_max // cp)
        kv_j = np.zeros((B, T_j, Dk), dtype=np.uint16)
        lens_j = np.zeros(B, dtype=np.int32)
        for b in range(B):
            own = np.arange(j, L[b], cp)
            kv_j[b, :own.size] = kv_full[b, own]
            lens_j[b] = own.size
        o, l = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv_j), torch.from_numpy(lens_j).cuda(), MLA_SCALE,
                                      n_split=n_split)
        parts += o
        part_l += l
    n_src = cp * n_split
    assert n_src <= 16 and H % n_src == 0
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    Hs = H // n_src
    # destination r of the merge = heads [r*Hs, (r+1)*Hs) of one contiguous output
    dcp.dcp_lse_reduce_ex(parts, part_l, n_src, B, H, 512, True, dcp.DCP_DTYPE_BF16,
                          [out.data_ptr() + r * Hs * 512 * 2 for r in range(n_src)],
                          [lse.data_ptr() + r * Hs * 4 for r in range(n_src)],
                          layout=dcp.Layout(src_row=H * 512, src_head=512, lse_row=H, lse_head=1,
                                            dst_row=H * 512, dst_head=512, lse_out_row=H))
    torch.cuda.synchronize()
    for b in range(B):
        o_ref, l_ref = attention(widen(q[b:b + 1]), widen(kv_full[b, :L[b]]), MLA_SCALE, dv=512)
        check_out(out[b:b + 1], o_ref, f"row {b}", kind="producer+merge")
        check_lse(lse[b:b + 1], l_ref, f"row {b}", kind="producer+merge")


def test_prefetch_flag_is_bit_identical_and_sees_fresh_inputs():
    """DCP_FLAG_PREFETCH brings Q and the first KV tile into L2 before the PDL
    wait, reading kv_len early for the addresses. Right after a kernel that
    rewrites the cache, kv_len and q (so the prefetch saw stale values), the
    results equal those of a plain call on the new inputs, bit for bit."""
    B, H, T = 4, 64, 600
    q1, kv1 = make_mla_inputs(B, H, T, 576, seed=31)
    q2, kv2 = make_mla_inputs(B, H, T, 576, seed=32)
    qd, kvd = dev_bf16(q1), dev_bf16(kv1)
    lens = torch.tensor([600, 300, 129, 5], dtype=torch.int32, device="cuda")
    lens2 = torch.tensor([450, 600, 1, 256], dtype=torch.int32, device="cuda")
    flags = dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH | dcp.DCP_MLA_FLAG_TCGEN05
    ref_o, ref_l = dcp.mla_decode_partial(dev_bf16(q2), dev_bf16(kv2), lens2, MLA_SCALE, n_split=2,
                                          flags=dcp.DCP_MLA_FLAG_TCGEN05)
    torch.cuda.synchronize()
    for _ in range(3):
        qd.copy_(dev_bf16(q1))
        kvd.copy_(dev_bf16(kv1))
        lens.copy_(torch.tensor([600, 300, 129, 5], dtype=torch.int32))
        torch.cuda.synchronize()
        # the copies below are the kernels right before the producer
        qd.copy_(dev_bf16(q2))
        kvd.copy_(dev_bf16(kv2))
        lens.copy_(lens2)
        o, l = dcp.mla_decode_partial(qd, kvd, lens, MLA_SCALE, n_split=2, flags=flags)
        torch.cuda.synchronize()
        for s_ in range(2):
            assert torch.equal(o[s_].view(torch.int16), ref_o[s_].view(torch.int16))
            assert torch.equal(l[s_].view(torch.int32), ref_l[s_].view(torch.int32))


def test_empty_shard_and_status_and_determinism():
    B, H, T = 2, 64, 80
    q, kv = make_mla_inputs(B, H, T, 576, seed=7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = torch.tensor([0, 80], dtype=torch.int32, device="cuda")
    o1, l1 = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), lens, MLA_SCALE, n_split=2, status=status)
    o2, l2 = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), lens, MLA_SCALE, n_split=2, status=status,
                                    flags=dcp.DCP_FLAG_PDL)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for s in range(2):
        assert (o1[s][0] == 0).all() and (l1[s][0] == -float("inf")).all()
        assert torch.equal(o1[s].view(torch.int16), o2[s].view(torch.int16))
        assert torch.equal(l1[s].view(torch.int32), l2[s].view(torch.int32))


def test_lengths_beyond_the_cache_are_clamped(oracle_mod):
    B, H, T = 2, 16, 40
    q, kv = make_mla_inputs(B, H, T, 576, seed=9)
    lens = np.array([1000, -3], dtype=np.int32)
    outs, lses = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), torch.from_numpy(lens).cuda(), MLA_SCALE)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_partials(q, kv, np.array([T, 0]), 1, MLA_SCALE, True)
    check_out(outs[0], ref_o[0], "clamped")
    check_lse(lses[0], ref_l[0], "clamped")


def test_graph_capture_of_producer_and_merge():
    B, H, T, cp = 2, 64, 128, 2
    q, kv = make_mla_inputs(B, H, T, 576, seed=11)
    qd, kvd = dev_bf16(q), dev_bf16(kv)
    lens = torch.tensor([128, 77], dtype=torch.int32, device="cuda")
    parts = [torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    pl = [torch.empty((B, H), dtype=torch.float32, device="cuda") for _ in range(cp)]
    outs = [torch.empty((B, H // cp, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    louts = [torch.empty((B, H // cp), dtype=torch.float32, device="cuda") for _ in range(cp)]

    def step():
        dcp.mla_decode_partial(qd, kvd, lens, MLA_SCALE, n_split=cp, outs=parts, lses=pl, flags=dcp.DCP_FLAG_PDL)
        dcp.merge(parts, pl, True, outs=outs, lse_outs=louts, flags=dcp.DCP_FLAG_PDL)

    step()
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(ref, outs))


def _interleaved_shards(kv_full, L, cp):
    """Shard j holds tokens j, j+cp, ... of every row (interleave 1)."""
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
        kvs.append(dev_bf16(kv_j))
        lens.append(torch.from_numpy(n_j).cuda())
    return kvs, lens


@pytest.mark.parametrize("kflags", KERNELS)
@pytest.mark.parametrize("cp,n_split,H,Dk", [(4, 2, 64, 576), (8, 2, 128, 576), (2, 4, 16, 512), (1, 16, 16, 576)])
def test_fused_dcp_decode_equals_full_attention(oracle_mod, cp, n_split, H, Dk, kflags):
    from oracle.attention import attention
    B, L_max = 3, 260
    q, kv_full = make_mla_inputs(B, H, L_max, Dk, seed=cp * 100 + n_split)
    L = np.array([L_max, 41, max(cp - 1, 1)], dtype=np.int32)
    kvs, lens = _interleaved_shards(kv_full, L, cp)
    outs, louts = dcp.mla_decode_dcp(dev_bf16(q), kvs, lens, MLA_SCALE, n_split=n_split, flags=kflags)
    torch.cuda.synchronize()
    Hl = H // cp
    for b in range(B):
        o_ref, l_ref = attention(widen(q[b:b + 1]), widen(kv_full[b, :L[b]]), MLA_SCALE, dv=512)
        for r in range(cp):
            check_out(outs[r][b:b + 1], o_ref[:, r * Hl:(r + 1) * Hl], f"row {b} dest {r}", kind="fused decode")
            check_lse(louts[r][b:b + 1], l_ref[:, r * Hl:(r + 1) * Hl], f"row {b} dest {r}", kind="fused decode")


def test_fused_dcp_decode_graph_replay_and_workspace_reuse():
    B, H, L_max, cp, n_split = 2, 64, 200, 4, 2
    q, kv_full = make_mla_inputs(B, H, L_max, 576, seed=3)
    kvs, lens = _interleaved_shards(kv_full, np.array([200, 150], dtype=np.int32), cp)
    qd = dev_bf16(q)
    ws = torch.empty((dcp.dcp_mla_decode_workspace_bytes(cp, n_split, B, H),), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((B, H // cp, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    louts = [torch.empty((B, H // cp), dtype=torch.float32, device="cuda") for _ in range(cp)]

    def call():
        dcp.mla_decode_dcp(qd, kvs, lens, MLA_SCALE, n_split=n_split, workspace=ws, outs=outs, lse_outs=louts,
                           flags=dcp.DCP_FLAG_PDL)

    call()
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs] + [l.clone() for l in louts]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
        call()  # the same workspace, in stream order
    for t in outs + louts:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    got = outs + louts
    assert all(torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
               for a, b in zip(ref, got))


@pytest.mark.parametrize("H", [16, 64, 128])
def test_tcgen05_and_mma_sync_kernels_agree(H):
    """Long ranges (many 128-token tiles, running-max moves) on both kernels."""
    B, T = 2, 2000
    q, kv = make_mla_inputs(B, H, T, 576, seed=H)
    # a drifting key scale makes later tiles' maxima exceed earlier ones (rescale path)
    kvf = widen(kv) * np.linspace(0.5, 1.5, T)[None, :, None]
    kv = bf16_bits(kvf.astype(np.float32))
    lens = torch.tensor([T, 1500], dtype=torch.int32, device="cuda")
    a_o, a_l = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), lens, MLA_SCALE, n_split=2,
                                      flags=dcp.DCP_MLA_FLAG_TCGEN05)
    b_o, b_l = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), lens, MLA_SCALE, n_split=2,
                                      flags=dcp.DCP_MLA_FLAG_MMA_SYNC)
    torch.cuda.synchronize()
    from oracle.attention import attention
    for s in range(2):
        for b, L in enumerate([T, 1500]):
            chunk = -(-L // 2)
            t0, t1 = s * chunk, min(L, (s + 1) * chunk)
            o_ref, l_ref = attention(widen(q[b:b + 1]), widen(kv[b, t0:t1]), MLA_SCALE, dv=512)
            check_out(a_o[s][b:b + 1], o_ref, f"tcgen05 split {s} row {b}")
            check_out(b_o[s][b:b + 1], o_ref, f"mma.sync split {s} row {b}")
            check_lse(a_l[s][b:b + 1], l_ref, f"tcgen05 split {s} row {b}")


@pytest.mark.parametrize("kflags", KERNELS)
@pytest.mark.parametrize("H,Dk", [(64, 576), (16, 512), (128, 576)])
def test_running_max_jumps_rescale_the_output(oracle_mod, H, Dk, kflags):
    """Single cached rows scaled up in later tiles: each spike lifts some heads'
    maxima by far more than 2^8 (base 2) above the running one, so the output
    accumulated so far must be rescaled (the lazy-rescale path of the tcgen05
    kernel, the per-tile rescale of the mma.sync kernel).

    Spikes are single tokens on purpose. A block of many scaled rows averages
    values of magnitude ~10-40 that cancel to ~0. There the 2^-9 relative
    rounding of each bf16 probability exceeds the absolute tolerance, and the
    two kernels agree bit for bit, so such a block tests the probability
    precision rather than the kernels."""
    B, T = 2, 1800
    q, kv = make_mla_inputs(B, H, T, Dk, seed=7 + H)
    kvf = widen(kv)
    for t, f in [(300, 4.0), (900, 8.0), (1700, 16.0)]:
        kvf[0, t] *= f
    for t, f in [(200, 6.0), (1000, 12.0)]:
        kvf[1, t] *= f
    kv = bf16_bits(kvf.astype(np.float32))
    lens = np.array([T, 1500], dtype=np.int32)
    for base_e in (True, False):
        outs, lses = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), torch.from_numpy(lens).cuda(), MLA_SCALE,
                                            lse_base_e=base_e, n_split=1, flags=kflags)
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_partials(q, kv, lens, 1, MLA_SCALE, base_e)
        check_out(outs[0], ref_o[0], f"H={H} base_e={base_e}")
        check_lse(lses[0], ref_l[0], f"H={H} base_e={base_e}")


@pytest.mark.parametrize("H,T,n_split", [(64, 1024, 4), (64, 500, 4), (32, 1024, 4), (32, 1024, 8), (16, 2048, 1),
                                         (128, 256, 2)])
def test_default_call_runs_the_kernel_the_query_names(H, T, n_split):
    """dcp_mla_decode_kernel names the kernel a default call launches: the
    default call's outputs equal, bit for bit, those of the call forcing it."""
    B = 3
    q, kv = make_mla_inputs(B, H, T, 576, seed=H + T + n_split)
    lens = torch.tensor([T, T - 7, 1], dtype=torch.int32, device="cuda")
    which = dcp.dcp_mla_decode_kernel(H, T, n_split)
    force = dcp.DCP_MLA_FLAG_TCGEN05 if which == dcp.DCP_MLA_KERNEL_TCGEN05 else dcp.DCP_MLA_FLAG_MMA_SYNC
    a_o, a_l = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), lens, MLA_SCALE, n_split=n_split)
    b_o, b_l = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), lens, MLA_SCALE, n_split=n_split, flags=force)
    torch.cuda.synchronize()
    for s in range(n_split):
        assert torch.equal(a_o[s], b_o[s]) and torch.equal(a_l[s], b_l[s]), f"split {s}"
    # and the other kernel rounds differently somewhere, so the identity above is not vacuous
    other = dcp.DCP_MLA_FLAG_MMA_SYNC if force == dcp.DCP_MLA_FLAG_TCGEN05 else dcp.DCP_MLA_FLAG_TCGEN05
    c_o, _ = dcp.mla_decode_partial(dev_bf16(q), dev_bf16(kv), lens, MLA_SCALE, n_split=n_split, flags=other)
    torch.cuda.synchronize()
    assert any(not torch.equal(a_o[s], c_o[s]) for s in range(n_split))


def test_picked_split_count_in_the_python_wrappers():
    """n_split=None picks dcp_mla_decode_pick_split's count; the results equal
    those of the explicit count, bit for bit."""
    B, H, T, cp = 4, 64, 1024, 2
    q, kv = make_mla_inputs(B, H, cp * T, 576, seed=5)
    kvs = [dev_bf16(kv[:, j * T:(j + 1) * T]) for j in range(cp)]
    lens = [torch.full((B,), T, dtype=torch.int32, device="cuda") for _ in range(cp)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = dcp.dcp_mla_decode_pick_split(cp, B, H, T, sms)
    assert n > 1
    a, al = dcp.mla_decode_dcp(dev_bf16(q), kvs, lens, MLA_SCALE, n_split=None)
    b, bl = dcp.mla_decode_dcp(dev_bf16(q), kvs, lens, MLA_SCALE, n_split=n)
    po, pl = dcp.mla_decode_partial(dev_bf16(q), kvs[0], lens[0], MLA_SCALE, n_split=None)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b)) and all(torch.equal(x, y) for x, y in zip(al, bl))
    assert len(po) == dcp.dcp_mla_decode_pick_split(1, B, H, T, sms)


@pytest.mark.parametrize("cp,n_split,H,B,L_max,base_e", [(8, 1, 128, 8, 4096, True), (4, 4, 64, 8, 4096, False),
                                                         (4, 2, 64, 3, 1100, True), (2, 1, 128, 5, 600, True)])
def test_one_kernel_decode_equals_two_launches_bit_for_bit(cp, n_split, H, B, L_max, base_e):
    """With DCP_MLA_FLAG_ONE_KERNEL dcp_mla_decode merges inside the
    producer's launch (one cooperative launch, a grid-wide sync, then every
    warp merges) when the tcgen05 grid fits one wave; by default the merge is
    its own launch. Same arithmetic in the same order: identical bits,
    including rows whose shards are partly or wholly empty."""
    q, kv_full = make_mla_inputs(B, H, L_max, 576, seed=cp * 1000 + H + B)
    L = np.full(B, L_max, dtype=np.int32)
    L[1] = L_max // 3
    L[2] = cp - 1  # one shard empty
    if B > 3:
        L[3] = 0   # every shard empty
    kvs, lens = _interleaved_shards(kv_full, L, cp)
    T = kvs[0].shape[1]
    tc = dcp.DCP_MLA_FLAG_TCGEN05
    assert dcp.dcp_mla_decode_kernel(H, T, n_split, tc) == dcp.DCP_MLA_KERNEL_TCGEN05
    qd = dev_bf16(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, l1 = dcp.mla_decode_dcp(qd, kvs, lens, MLA_SCALE, n_split=n_split, lse_base_e=base_e, status=status,
                                flags=tc | dcp.DCP_FLAG_PDL | dcp.DCP_MLA_FLAG_ONE_KERNEL)
    o2, l2 = dcp.mla_decode_dcp(qd, kvs, lens, MLA_SCALE, n_split=n_split, lse_base_e=base_e, status=status,
                                flags=tc | dcp.DCP_FLAG_PDL)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for r in range(cp):
        assert torch.equal(o1[r].view(torch.int16), o2[r].view(torch.int16)), f"destination {r} output"
        assert torch.equal(l1[r].view(torch.int32), l2[r].view(torch.int32)), f"destination {r} LSE"
    if B > 3:
        assert all(bool((o[3] == 0).all()) and bool((l[3] == -float("inf")).all()) for o, l in zip(o1, l1))


def test_one_kernel_decode_matches_attention_and_replays_in_a_graph(oracle_mod):
    from oracle.attention import attention
    B, H, L_max, cp, n_split = 3, 64, 900, 4, 1
    q, kv_full = make_mla_inputs(B, H, L_max, 576, seed=77)
    L = np.array([900, 513, 129], dtype=np.int32)
    kvs, lens = _interleaved_shards(kv_full, L, cp)
    qd = dev_bf16(q)
    flags = dcp.DCP_MLA_FLAG_TCGEN05 | dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH | dcp.DCP_MLA_FLAG_ONE_KERNEL
    ws = torch.empty((dcp.dcp_mla_decode_workspace_bytes(cp, n_split, B, H),), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((B, H // cp, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    louts = [torch.empty((B, H // cp), dtype=torch.float32, device="cuda") for _ in range(cp)]

    def call():
        dcp.mla_decode_dcp(qd, kvs, lens, MLA_SCALE, n_split=n_split, workspace=ws, outs=outs, lse_outs=louts,
                           flags=flags)

    call()
    torch.cuda.synchronize()
    Hl = H // cp
    for b in range(B):
        o_ref, l_ref = attention(widen(q[b:b + 1]), widen(kv_full[b, :L[b]]), MLA_SCALE, dv=512)
        for r in range(cp):
            check_out(outs[r][b:b + 1], o_ref[:, r * Hl:(r + 1) * Hl], f"row {b} dest {r}", kind="fused decode")
            check_lse(louts[r][b:b + 1], l_ref[:, r * Hl:(r + 1) * Hl], f"row {b} dest {r}", kind="fused decode")
    ref = [o.clone() for o in outs] + [l.clone() for l in louts]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
        call()
    for t in outs + louts:
        t.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(ref, outs + louts))


@pytest.mark.parametrize("kflags", KERNELS)
def test_a_wait_that_never_completes_gives_up_and_reports(oracle_mod, kflags):
    """The bounded waits, exercised on the GPU without a fault: with the stall
    test flag every CTA arms its first KV tile's barrier for 16 bytes that
    never arrive. Each such wait gives up after 20 ms, the status word reads 1,
    the call ends (no hang, well under the two-second limit of a normal call),
    a CTA whose range is empty still writes its zero output, and the context
    stays usable: the same call without the flag then matches the oracle."""
    import time

    B, H, T, n_split = 3, 64, 600, 2
    q, kv = make_mla_inputs(B, H, T, 576, seed=11)
    lens = np.array([T, 0, 300], dtype=np.int32)
    qd, kvd, ld = dev_bf16(q), dev_bf16(kv), torch.from_numpy(lens).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    outs, lses = dcp.mla_decode_partial(qd, kvd, ld, MLA_SCALE, n_split=n_split, status=status,
                                        flags=kflags | dcp.DCP_MLA_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == 1
    assert elapsed < 1.5, f"the stalled call took {elapsed:.2f} s"
    for s in range(n_split):
        assert (outs[s][1] == 0).all() and (lses[s][1] == -float("inf")).all()

    status.zero_()
    outs, lses = dcp.mla_decode_partial(qd, kvd, ld, MLA_SCALE, n_split=n_split, status=status, flags=kflags)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle_partials(q, kv, lens, n_split, MLA_SCALE, True)
    for s in range(n_split):
        check_out(outs[s], ref_o[s], f"split {s} after a stalled call")
        check_lse(lses[s], ref_l[s], f"split {s} after a stalled call")


@pytest.mark.parametrize("one_kernel", [False, True])
def test_fused_decode_after_a_stalled_producer(oracle_mod, one_kernel):
    """dcp_mla_decode with the stall test flag: the producer's waits give up,
    the status word reads 1 and the call ends, with the merge as a second
    launch or, with the one-kernel flag, after the grid-wide sync that every
    CTA of an aborted producer still reaches. A normal call follows and
    matches attention over the whole context."""
    from oracle.attention import attention

    cp, n_split, B, H, T = 2, 2, 2, 64, 512
    q, kv0 = make_mla_inputs(B, H, T, 576, seed=21)
    _, kv1 = make_mla_inputs(B, H, T, 576, seed=22)
    lens = [np.array([T, 200], dtype=np.int32), np.array([300, 0], dtype=np.int32)]
    qd = dev_bf16(q)
    kvs = [dev_bf16(kv0), dev_bf16(kv1)]
    lds = [torch.from_numpy(x).cuda() for x in lens]
    extra = dcp.DCP_MLA_FLAG_ONE_KERNEL if one_kernel else 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dcp.mla_decode_dcp(qd, kvs, lds, MLA_SCALE, n_split=n_split, status=status,
                       flags=dcp.DCP_MLA_FLAG_TCGEN05 | dcp.DCP_MLA_FLAG_TEST_STALL | extra)
    torch.cuda.synchronize()
    assert int(status.item()) == 1

    status.zero_()
    outs, lse_outs = dcp.mla_decode_dcp(qd, kvs, lds, MLA_SCALE, n_split=n_split, status=status,
                                        flags=dcp.DCP_MLA_FLAG_TCGEN05 | extra)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qf, kvf = widen(q), [widen(kv0), widen(kv1)]
    Hl = H // cp
    for b in range(B):
        ctx = np.concatenate([kvf[j][b, :lens[j][b]] for j in range(cp)], axis=0)
        o, l = attention(qf[b:b + 1], ctx, MLA_SCALE, True, 512)
        for r in range(cp):
            check_out(outs[r][b], o[0, r * Hl:(r + 1) * Hl], f"row {b} dest {r}", kind="fused decode")
            check_lse(lse_outs[r][b], l[0, r * Hl:(r + 1) * Hl], f"row {b} dest {r}", kind="fused decode")


@pytest.mark.parametrize("H,T,kflags", [(16, 5, dcp.DCP_MLA_FLAG_MMA_SYNC), (64, 128, dcp.DCP_MLA_FLAG_TCGEN05)])
def test_producer_at_the_largest_batch(oracle_mod, H, T, kflags):
    """B = 65535 rows, the producer's largest batch (one grid row per batch
    row): every row is computed (LSEs finite where the row has tokens, -inf
    where it has none), and sampled rows, the last ones included, match the
    oracle attention. Inputs are drawn on the device by a seeded generator;
    the sampled rows are copied to the host for the oracle."""
    B, Dk = 65535, 576
    gen = torch.Generator(device="cuda")
    gen.manual_seed(H + T)
    q = torch.randn((B, H, Dk), generator=gen, device="cuda").to(torch.bfloat16)
    kv = torch.randn((B, T, Dk), generator=gen, device="cuda").to(torch.bfloat16)
    lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
    lens[::7] = 0
    outs, lses = dcp.mla_decode_partial(q, kv, lens, MLA_SCALE, n_split=1, flags=kflags)
    torch.cuda.synchronize()
    empty = lens == 0
    assert torch.isfinite(lses[0][~empty]).all() and (lses[0][empty] == -float("inf")).all()
    assert not torch.isnan(outs[0].float()).any()
    rows = [1, 2, 1000, 40001, B - 2, B - 1]
    for b in rows:
        qb = q[b:b + 1].view(torch.int16).cpu().numpy().view(np.uint16)
        kvb = kv[b:b + 1].view(torch.int16).cpu().numpy().view(np.uint16)
        lb = lens[b:b + 1].cpu().numpy()
        ref_o, ref_l = oracle_partials(qb, kvb, lb, 1, MLA_SCALE, True)
        check_out(outs[0][b:b + 1], ref_o[0], f"row {b}")
        check_lse(lses[0][b:b + 1], ref_l[0], f"row {b}")


def test_concurrent_callers_on_their_own_streams():
    """Two host threads call the producer, the fused decode and the merge at
    the same time, each on its own stream (ctypes releases the GIL during a
    call, so the library runs concurrently on both). Every result equals the
    single-threaded one bit for bit."""
    import threading

    B, H, T, cp = 3, 64, 600, 2
    q, kv = make_mla_inputs(B, H, T, 576, seed=31)
    qd, kvd = dev_bf16(q), dev_bf16(kv)
    lens = torch.tensor([T, 300, 0], dtype=torch.int32, device="cuda")
    shard_lens = [lens, torch.tensor([T, 1, 0], dtype=torch.int32, device="cuda")]

    def work(stream):
        with torch.cuda.stream(stream):
            o, l = dcp.mla_decode_partial(qd, kvd, lens, MLA_SCALE, n_split=2, stream=stream)
            fo, fl = dcp.mla_decode_dcp(qd, [kvd, kvd], shard_lens, MLA_SCALE, n_split=2, stream=stream)
            mo, ml = dcp.merge(o, l, True, stream=stream)
        stream.synchronize()
        return [x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32) for x in o + l + fo + fl + mo + ml]

    torch.cuda.synchronize()  # inputs in place before other streams read them
    ref = work(torch.cuda.Stream())
    results, errors = {}, []

    def run(k):
        try:
            s = torch.cuda.Stream()
            for it in range(20):
                got = work(s)
                if not all(torch.equal(a, b) for a, b in zip(ref, got)):
                    results[k] = f"mismatch at iteration {it}"
                    return
            results[k] = "ok"
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert results == {0: "ok", 1: "ok"}, results


@pytest.mark.parametrize("kflags", KERNELS)
def test_empty_cache_gives_zero_outputs_and_neg_inf(kflags):
    """T = 0 (a cache that holds no tokens for any row): every split writes
    output 0 and LSE -inf, whatever the token counts say (they clamp to 0).
    And a fused decode in which one shard has no tokens for any row equals
    the producer over the other shard alone, bit for bit (weights 0 and 1)."""
    B, H = 3, 64
    q, kv = make_mla_inputs(B, H, 300, 576, seed=41)
    qd, kvd = dev_bf16(q), dev_bf16(kv)
    lens = torch.tensor([5, 0, 100], dtype=torch.int32, device="cuda")
    outs = [torch.full((B, H, 512), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    lses = [torch.zeros((B, H), dtype=torch.float32, device="cuda") for _ in range(2)]
    # the C entry point with T = 0 (the cache pointer is valid but no row of it is read)
    dcp.dcp_mla_decode_partial(qd, kvd, lens, B, H, 576, 512, 0, MLA_SCALE, True, 2, outs, lses, flags=kflags)
    torch.cuda.synchronize()
    for s_ in range(2):
        assert (outs[s_] == 0).all() and (lses[s_] == -float("inf")).all()

    none = torch.zeros((B,), dtype=torch.int32, device="cuda")
    full = torch.full((B,), 300, dtype=torch.int32, device="cuda")
    _, kv2 = make_mla_inputs(B, H, 300, 576, seed=42)
    both, both_l = dcp.mla_decode_dcp(qd, [dev_bf16(kv2), kvd], [none, full], MLA_SCALE, n_split=1, flags=kflags)
    alone, alone_l = dcp.mla_decode_partial(qd, kvd, full, MLA_SCALE, n_split=1, flags=kflags)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(both, dim=1).view(torch.int16), alone[0].view(torch.int16))
    assert torch.equal(torch.cat(both_l, dim=1).view(torch.int32), alone_l[0].view(torch.int32))


@pytest.mark.parametrize("flags", [dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH, dcp.DCP_MLA_FLAG_ONE_KERNEL,
                                   dcp.DCP_MLA_FLAG_MMA_SYNC])
def test_no_alloc_decode_is_bit_identical_to_the_workspace_decode_under_each_flag(flags):
    """The built-in scratch only replaces the caller's workspace: with the
    launch flags, the one-kernel form and the mma.sync producer, the
    no-allocation decode gives the same bits as dcp_mla_decode."""
    cp, n_split, B, H, T = 2, 2, 3, 64, 300
    q, kv0 = make_mla_inputs(B, H, T, 576, seed=61)
    _, kv1 = make_mla_inputs(B, H, T, 576, seed=62)
    qd, kvs = dev_bf16(q), [dev_bf16(kv0), dev_bf16(kv1)]
    lens = [torch.tensor([T, 17, 0], dtype=torch.int32, device="cuda"),
            torch.tensor([200, 0, 0], dtype=torch.int32, device="cuda")]
    ws = torch.empty((dcp.dcp_mla_decode_workspace_bytes(cp, n_split, B, H),), dtype=torch.uint8, device="cuda")
    outs = [[torch.empty((B, H // cp, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)] for _ in range(2)]
    louts = [[torch.empty((B, H // cp), dtype=torch.float32, device="cuda") for _ in range(cp)] for _ in range(2)]
    dcp.dcp_mla_decode(qd, kvs, lens, cp, B, H, 576, 512, T, MLA_SCALE, True, n_split, ws, ws.numel(), outs[0],
                       louts[0], flags=flags)
    dcp.dcp_mla_decode_noalloc(qd, kvs, lens, cp, B, H, 576, 512, T, MLA_SCALE, True, n_split, outs[1], louts[1],
                               flags=flags)
    torch.cuda.synchronize()
    for r in range(cp):
        assert torch.equal(outs[0][r].view(torch.int16), outs[1][r].view(torch.int16))
        assert torch.equal(louts[0][r].view(torch.int32), louts[1][r].view(torch.int32))
