"""GPU parity: the sm_103a kernel, called through the C ABI, against the CPU
oracle on the same seeded inputs.

Tolerances (bf16 outputs): |gpu - ref| <= 1e-2 + 8e-3*|ref| element-wise, and
the tighter bound half a bf16 ulp plus fp32 accumulation error,
|gpu - ref| <= 2^-8*|ref| + 1e-5 (round-to-nearest-even from an fp32 sum).
Merged LSE: |gpu - ref| <= 1e-5 * max(|ref|, 1); -inf exactly where the oracle
has -inf. Every output buffer sits between guard bands that must survive.
"""
import math

import numpy as np
import pytest
import torch

import decode_context_mla_dcp_gb300 as dcp
from decode_context_mla_dcp_gb300 import build as dcp_build
from decode_context_mla_dcp_gb300.inputs import BF16_QNAN, CONFIGS, bf16_bits, make_merge_inputs, tiny_qkv

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 8e-3
TIGHT_R, TIGHT_A = 2.0 ** -8, 1e-5
LSE_R = 1e-5
GUARD = 256          # bytes on each side of an output
SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    dcp_build.build()
    dcp.load()
    torch.cuda.set_device(0)
    yield


# ---- helpers -------------------------------------------------------------------

def to_dev_bits(a: np.ndarray, dtype=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype).cuda()


class Guarded:
    """A device buffer of n elements between two guard bands of SENTINEL bytes."""

    def __init__(self, shape, dtype):
        self.n = int(np.prod(shape)) if len(shape) else 1
        self.esize = torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD * 2 + self.n * self.esize,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.n * self.esize].view(dtype).view(shape)

    def guards_ok(self):
        g = torch.cat([self.raw[:GUARD], self.raw[GUARD + self.n * self.esize:]])
        return bool((g == SENTINEL).all())


def run_gpu(inp, flags=0, dtype=torch.bfloat16, write_lse=True):
    cp, B, H, D = inp.cp, inp.B, inp.H, inp.D
    Hl = H // cp
    srcs = [to_dev_bits(s, dtype) for s in inp.srcs]
    lses = [torch.from_numpy(np.ascontiguousarray(l)).cuda() for l in inp.lses]
    outs = [Guarded((B, Hl, D), dtype) for _ in range(cp)]
    louts = [Guarded((B, Hl), torch.float32) for _ in range(cp)]
    dcp.dcp_lse_reduce_ex([s.data_ptr() for s in srcs], [l.data_ptr() for l in lses], cp, B, H, D,
                          inp.lse_base_e, dcp.DCP_DTYPE_F16 if dtype == torch.float16 else dcp.DCP_DTYPE_BF16,
                          [o.t.data_ptr() for o in outs],
                          [l.t.data_ptr() for l in louts] if write_lse else None,
                          layout=dcp.Layout(src_row=H * D, src_head=D, lse_row=inp.lse_stride, lse_head=1,
                                            dst_row=Hl * D, dst_head=D, lse_out_row=Hl),
                          flags=flags)
    torch.cuda.synchronize()
    for g in outs + louts:
        assert g.guards_ok(), "a write landed outside an output buffer"
    return ([o.t.float().double().cpu().numpy() for o in outs],
            [l.t.double().cpu().numpy() for l in louts] if write_lse else None)


def assert_out_close(got, ref, what=""):
    assert not np.isnan(got).any(), f"{what}: NaN in GPU output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} elements outside atol/rtol; max err {err.max():.3g}"
    tight = err > TIGHT_R * np.abs(ref) + TIGHT_A
    assert not tight.any(), f"{what}: {tight.sum()} elements beyond half a bf16 ulp; max err {err.max():.3g}"


def assert_lse_close(got, ref, what=""):
    ninf = ref == -np.inf
    assert np.array_equal(got == -np.inf, ninf), f"{what}: -inf pattern differs"
    assert not np.isnan(got).any()
    g, r = got[~ninf], ref[~ninf]
    err = np.abs(g - r)
    assert (err <= LSE_R * np.maximum(np.abs(r), 1.0)).all(), f"{what}: LSE max err {err.max() if err.size else 0:.3g}"


def check_against_oracle(oracle_mod, inp, flags=0, dtype=torch.bfloat16, what=""):
    outs, louts = run_gpu(inp, flags=flags, dtype=dtype)
    ref, lref = oracle_mod.merge(inp.srcs, [l.reshape(inp.B, -1) for l in inp.lses], inp.lse_base_e,
                                 dtype="f16" if dtype == torch.float16 else "bf16", H=inp.H,
                                 src_strides=(inp.H * inp.D, inp.D), lse_strides=(inp.lse_stride, 1))
    for r in range(inp.cp):
        if dtype == torch.float16:
            err = np.abs(outs[r] - ref[r])
            assert (err <= 2.0 ** -11 * np.abs(ref[r]) + 1e-5).all(), f"{what} fp16 dest {r}"
        else:
            assert_out_close(outs[r], ref[r], f"{what} dest {r}")
        assert_lse_close(louts[r], lref[r], f"{what} dest {r}")
    return outs, louts


# ---- the configs ---------------------------------------------------------------

def test_tiny_exactness_matches_full_attention(oracle_mod):
    from oracle.attention import attention, split_partials
    q, kv = tiny_qkv(0)
    scale = 1.0 / math.sqrt(512)
    o_parts, l_parts = split_partials(q, kv, [np.arange(0, 32), np.arange(32, 64)], scale)
    o_full, l_full = attention(q, kv, scale)

    class Inp:
        pass
    inp = Inp()
    inp.cp, inp.B, inp.H, inp.D, inp.lse_base_e, inp.lse_stride = 2, 3, 16, 512, True, 16
    inp.srcs = [bf16_bits(o.astype(np.float32)) for o in o_parts]
    inp.lses = [l.astype(np.float32) for l in l_parts]
    outs, louts = check_against_oracle(oracle_mod, inp, what="tiny")
    got = np.concatenate(outs, axis=1)
    err = np.abs(got - o_full)
    assert (err <= ATOL + RTOL * np.abs(o_full)).all(), f"tiny vs full attention: max err {err.max():.3g}"
    lg = np.concatenate(louts, axis=1)
    assert (np.abs(lg - l_full) <= LSE_R * np.maximum(np.abs(l_full), 1)).all()


@pytest.mark.parametrize("rows", CONFIGS["kimi"].rows)
def test_kimi_config(oracle_mod, rows):
    check_against_oracle(oracle_mod, make_merge_inputs("kimi", rows, seed=0), what=f"kimi B={rows}")


@pytest.mark.parametrize("rows", CONFIGS["deepseek"].rows)
def test_deepseek_config(oracle_mod, rows):
    check_against_oracle(oracle_mod, make_merge_inputs("deepseek", rows, seed=0), what=f"deepseek B={rows}")


@pytest.mark.parametrize("flags", [0, dcp.DCP_FLAG_PRELOAD, dcp.DCP_FLAG_LSE_FIRST])
def test_spec_decode_config_with_empty_shards(oracle_mod, flags):
    inp = make_merge_inputs("spec", 1024, seed=0)
    assert inp.empty.any()
    check_against_oracle(oracle_mod, inp, flags=flags, what="spec")


def test_stress_config_full_size_sampled(oracle_mod):
    """4096 rows x 128 heads x cp 8: the full launch the benchmark times.
    The oracle checks 48 sampled rows element by element; every element is
    checked for the properties that hold at any size (finite, inside the
    sources' range)."""
    inp = make_merge_inputs("stress", 4096, seed=0)
    cp, B, H, D = inp.cp, inp.B, inp.H, inp.D
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    outs, louts = dcp.merge(srcs, lses, True)
    torch.cuda.synchronize()
    full = torch.cat(outs, dim=1).float()                      # [B, H, D]
    stack = torch.stack([s.float() for s in srcs])             # [cp, B, H, D]
    assert torch.isfinite(full).all()
    lo, hi = stack.min(0).values, stack.max(0).values
    slack = 2.0 ** -8 * torch.maximum(lo.abs(), hi.abs()) + 1e-6
    assert bool(((full >= lo - slack) & (full <= hi + slack)).all())
    del stack
    rng = np.random.default_rng(123)
    rows = np.sort(rng.choice(B, size=48, replace=False))
    rows = np.unique(np.concatenate([rows, [0, B - 1]]))
    sub_srcs = [s[rows] for s in inp.srcs]
    sub_lses = [l[rows] for l in inp.lses]
    ref, lref = oracle_mod.merge(sub_srcs, sub_lses, True)
    idx = torch.from_numpy(rows).cuda()
    for r in range(cp):
        assert_out_close(outs[r][idx].float().double().cpu().numpy(), ref[r], f"stress dest {r}")
        assert_lse_close(louts[r][idx].double().cpu().numpy(), lref[r], f"stress dest {r}")


# ---- odd shapes and edge cases ----------------------------------------------------

@pytest.mark.parametrize("cp,H", [(1, 3), (2, 2), (3, 9), (5, 10), (7, 7), (8, 24), (9, 18), (16, 32)])
@pytest.mark.parametrize("B", [1, 3, 49])
def test_odd_shapes(oracle_mod, cp, H, B):
    inp = make_merge_inputs("deepseek", B, seed=cp * 100 + B, cp=cp, H=H)
    check_against_oracle(oracle_mod, inp, what=f"cp={cp} H={H} B={B}")


@pytest.mark.parametrize("D", [8, 64, 256, 520, 1024, 1040])
def test_head_widths(oracle_mod, D):
    inp = make_merge_inputs("kimi", 7, seed=D, cp=4, H=8, D=D)
    check_against_oracle(oracle_mod, inp, what=f"D={D}")


@pytest.mark.parametrize("flags", [dcp.DCP_FLAG_PRELOAD, dcp.DCP_FLAG_LSE_FIRST, dcp.DCP_FLAG_PDL])
@pytest.mark.parametrize("cp", [2, 4, 8, 12])
def test_schedules(oracle_mod, flags, cp):
    inp = make_merge_inputs("spec", 64, seed=cp, cp=cp, H=cp * 4, p_empty=0.3)
    check_against_oracle(oracle_mod, inp, flags=flags, what=f"flags={flags} cp={cp}")


def test_fp16(oracle_mod):
    inp = make_merge_inputs("spec", 33, seed=5, dtype="f16", cp=4, H=16)
    check_against_oracle(oracle_mod, inp, dtype=torch.float16, what="fp16")


def test_rows_with_every_source_empty(oracle_mod):
    inp = make_merge_inputs("kimi", 9, seed=2, cp=4, H=8)
    for j in range(4):
        inp.lses[j][[0, 4, 8]] = -np.inf
        inp.srcs[j][[0, 4, 8]] = BF16_QNAN
    outs, louts = check_against_oracle(oracle_mod, inp, what="empty rows")
    for r in range(4):
        assert np.array_equal(outs[r][[0, 4, 8]], np.zeros_like(outs[r][[0, 4, 8]]))
        assert (louts[r][[0, 4, 8]] == -np.inf).all()


def test_single_live_source_is_copied_bit_exact():
    # One finite LSE per (row, head): weight exactly 1, so bf16 -> fp32 -> bf16
    # round-trips and the output equals that source's row bit for bit.
    inp = make_merge_inputs("kimi", 5, seed=9, cp=4, H=8)
    live = np.random.default_rng(0).integers(0, 4, size=(5, 8))
    for j in range(4):
        inp.lses[j][live != j] = -np.inf
    outs, _ = run_gpu(inp)
    for r in range(4):
        for b in range(5):
            for i in range(2):
                h = r * 2 + i
                src = (inp.srcs[live[b, h]][b, h].astype(np.uint32) << 16).view(np.float32)
                assert np.array_equal(outs[r][b, i], src.astype(np.float64))


def test_lse_stride_and_null_lse_outputs(oracle_mod):
    inp = make_merge_inputs("deepseek", 6, seed=4, cp=4, H=8)
    # padded LSE rows (stride 13) with NaN padding
    pad = []
    for l in inp.lses:
        p = np.full((6, 13), np.nan, dtype=np.float32)
        p[:, :8] = l.reshape(6, 8)
        pad.append(p)
    inp.lses, inp.lse_stride = pad, 13
    check_against_oracle(oracle_mod, inp, what="lse stride 13")
    outs, louts = run_gpu(inp, write_lse=False)
    assert louts is None


@pytest.mark.parametrize("s_q", [2, 4])
@pytest.mark.parametrize("flags", [0, dcp.DCP_FLAG_PRELOAD, dcp.DCP_FLAG_LSE_FIRST,
                                   dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH])
def test_flashmla_lse_head_stride(oracle_mod, s_q, flags):
    # FlashMLA with s_q query tokens per row: partial outputs [B, s_q, H, D],
    # LSEs [B, H, s_q]. One call per token t: sources start t*H*D elements in
    # with row stride s_q*H*D; LSEs start t elements in with row stride H*s_q
    # and head stride s_q; destinations are [B, s_q, H/cp, D] and merged LSEs
    # [B, s_q, H/cp]. Checked element by element against the oracle called
    # with the same strides ("[DCP] Run fi_a2a on FlashInfer's fused
    # all-to-all + LSE reduce", "Accuracy Tests": FlashMLA's LSE layout).
    B, cp, H, D = 9, 8, 128, 512
    Hl = H // cp
    inp = make_merge_inputs("deepseek", B * s_q, seed=40 + s_q)
    src_full = [s.reshape(B, s_q, H, D) for s in inp.srcs]
    lse_full = [np.ascontiguousarray(l.reshape(B, s_q, H).transpose(0, 2, 1)) for l in inp.lses]  # [B, H, s_q]
    srcs = [to_dev_bits(s) for s in src_full]
    lses = [torch.from_numpy(l).cuda() for l in lse_full]
    outs = [Guarded((B, s_q, Hl, D), torch.bfloat16) for _ in range(cp)]
    louts = [Guarded((B, s_q, Hl), torch.float32) for _ in range(cp)]
    lay = dcp.Layout(src_row=s_q * H * D, src_head=D, lse_row=H * s_q, lse_head=s_q,
                     dst_row=s_q * Hl * D, dst_head=D, lse_out_row=s_q * Hl)
    for t in range(s_q):
        dcp.dcp_lse_reduce_ex([x.data_ptr() + t * H * D * 2 for x in srcs], [x.data_ptr() + t * 4 for x in lses],
                              cp, B, H, D, True, dcp.DCP_DTYPE_BF16,
                              [o.t.data_ptr() + t * Hl * D * 2 for o in outs],
                              [o.t.data_ptr() + t * Hl * 4 for o in louts], layout=lay, flags=flags)
    torch.cuda.synchronize()
    for g in outs + louts:
        assert g.guards_ok(), "a write landed outside an output buffer"
    for t in range(s_q):
        ref, lref = oracle_mod.merge([np.ascontiguousarray(s[:, t]) for s in src_full],
                                     [l.reshape(-1)[t:] for l in lse_full], True, H=H, D=D,
                                     lse_strides=(H * s_q, s_q))
        for r in range(cp):
            assert_out_close(outs[r].t[:, t].float().double().cpu().numpy(), ref[r], f"s_q={s_q} t={t} dest {r}")
            assert_lse_close(louts[r].t[:, t].double().cpu().numpy(), lref[r], f"s_q={s_q} t={t} dest {r}")


def test_strided_layouts(oracle_mod):
    # padded token stride for sources, a wider head backing array, and padded
    # destinations, through the tensor-level entry point
    B, H, D, cp = 5, 8, 512, 4
    inp = make_merge_inputs("kimi", B, seed=8, cp=cp, H=H)
    wide = []
    for s in inp.srcs:
        w = np.full((B, H, D + 64), BF16_QNAN, dtype=np.uint16)
        w[:, :, :D] = s
        wide.append(to_dev_bits(w)[:, :, :D])
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    dst_back = [torch.zeros((B, H // cp + 1, D + 8), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    outs = [d[:, 1:, :D] for d in dst_back]
    outs, louts = dcp.merge(wide, lses, False, outs=outs)
    torch.cuda.synchronize()
    ref, lref = oracle_mod.merge(inp.srcs, inp.lses, False)
    for r in range(cp):
        assert_out_close(outs[r].float().double().cpu().numpy(), ref[r], f"strided dest {r}")
        assert (dst_back[r][:, 0] == 0).all() and (dst_back[r][:, :, D:] == 0).all()


@pytest.mark.parametrize("cfg,interleave", [("kimi", 1), ("kimi", 16), ("deepseek", 1), ("deepseek", 64)])
@pytest.mark.parametrize("flags", [0, dcp.DCP_FLAG_PRELOAD, dcp.DCP_FLAG_LSE_FIRST])
def test_seq_len_masking(oracle_mod, cfg, interleave, flags):
    # Context lengths around every shard boundary (L <= j*interleave empties
    # shard j), including 0. Empty shards' LSE entries hold NaN and their
    # payloads NaN: both must be ignored.
    inp = make_merge_inputs(cfg, 40, seed=interleave)
    cp, B, H = inp.cp, inp.B, inp.H
    rng = np.random.default_rng(interleave)
    lens = rng.integers(0, cp * interleave + 3, size=B).astype(np.int32)
    lens[:4] = [0, 1, interleave, cp * interleave]
    for j in range(cp):
        empty = lens <= j * interleave
        inp.lses[j] = inp.lses[j].copy()
        inp.lses[j].reshape(B, H)[empty] = np.nan
        inp.srcs[j][empty] = BF16_QNAN
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    sl = torch.from_numpy(lens).cuda()
    outs, louts = dcp.merge(srcs, lses, inp.lse_base_e, seq_lens=sl, interleave=interleave, flags=flags)
    torch.cuda.synchronize()
    ref, lref = oracle_mod.merge(inp.srcs, [l.reshape(B, H) for l in inp.lses], inp.lse_base_e, seq_lens=lens,
                                 interleave=interleave)
    for r in range(cp):
        assert_out_close(outs[r].float().double().cpu().numpy(), ref[r], f"masked dest {r}")
        assert_lse_close(louts[r].double().cpu().numpy(), lref[r], f"masked dest {r}")
    # L = 0 rows
    for r in range(cp):
        assert (outs[r][0] == 0).all() and (louts[r][0] == -float("inf")).all()


def test_seq_len_masking_matches_split_attention_over_row_contexts(oracle_mod):
    # Partials from fp64 attention over each row's interleaved shards, rounded
    # to bf16; the masked GPU merge must reproduce attention over the row's
    # whole context.
    from tests.test_oracle_pins import _masked_case
    cp, interleave, lens = 4, 4, [3, 9, 17]
    srcs64, lses64, o_full, l_full = _masked_case(cp, interleave, lens)
    srcs = [to_dev_bits(bf16_bits(np.nan_to_num(s, nan=0.0).astype(np.float32))) for s in srcs64]
    lses = [torch.from_numpy(l.astype(np.float32)).cuda() for l in lses64]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    outs, louts = dcp.merge(srcs, lses, True, seq_lens=sl, interleave=interleave)
    torch.cuda.synchronize()
    got = torch.cat(outs, 1).float().double().cpu().numpy()
    assert (np.abs(got - o_full) <= ATOL + RTOL * np.abs(o_full)).all()
    lg = torch.cat(louts, 1).double().cpu().numpy()
    assert (np.abs(lg - l_full) <= LSE_R * np.maximum(np.abs(l_full), 1)).all()


def test_empty_batch_writes_nothing():
    inp = make_merge_inputs("kimi", 1, seed=0)
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    g = [Guarded((1, 16, 512), torch.bfloat16) for _ in range(4)]
    dcp.dcp_lse_reduce(srcs, lses, 64, 4, 0, 64, 512, False, [x.t for x in g])
    torch.cuda.synchronize()
    assert all(bool((x.raw == SENTINEL).all()) for x in g)


def test_misaligned_device_pointer_is_rejected_before_launch():
    inp = make_merge_inputs("kimi", 1, seed=0)
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    outs = [torch.empty((1, 16, 512), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    with pytest.raises(dcp.DcpError) as e:
        dcp.dcp_lse_reduce([srcs[0].data_ptr() + 2] + srcs[1:], lses, 64, 4, 1, 64, 512, False, outs)
    assert e.value.status == -6


# ---- determinism, graphs, streams ---------------------------------------------------

def _bits(ts):
    return [t.view(torch.int16).clone() if t.dtype != torch.float32 else t.view(torch.int32).clone() for t in ts]


def test_bit_identical_across_calls_schedules_and_pdl():
    inp = make_merge_inputs("spec", 256, seed=1)
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    base_o, base_l = dcp.merge(srcs, lses, True)
    ref = _bits(base_o) + _bits(base_l)
    pf = dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH
    for flags in [0, 0, dcp.DCP_FLAG_PRELOAD, dcp.DCP_FLAG_LSE_FIRST, dcp.DCP_FLAG_PDL,
                  dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PRELOAD, pf, pf | dcp.DCP_FLAG_PRELOAD,
                  pf | dcp.DCP_FLAG_LSE_FIRST, dcp.DCP_FLAG_PREFETCH]:
        o, l = dcp.merge(srcs, lses, True, flags=flags)
        got = _bits(o) + _bits(l)
        assert all(torch.equal(a, b) for a, b in zip(ref, got)), f"flags={flags}"


def test_prefetch_before_the_wait_sees_the_previous_kernels_writes():
    # Merge A writes outputs that merge B reads as its sources and LSEs. With
    # PDL, B's CTAs start while A runs and prefetch those lines into L2 before
    # A has written them (they hold NaN then); after its wait B must read A's
    # values. Compared bit for bit with the same chain run without PDL or
    # prefetch, 20 times over.
    B, H, cp = 64, 32, 2
    inp = make_merge_inputs("kimi", B, seed=31, cp=cp, H=H)
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    mid = [torch.empty((B, H // cp, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    mid_l = [torch.empty((B, H // cp), dtype=torch.float32, device="cuda") for _ in range(cp)]
    fin = [torch.empty((B, H // (2 * cp), 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    fin_l = [torch.empty((B, H // (2 * cp)), dtype=torch.float32, device="cuda") for _ in range(cp)]

    flush = torch.zeros((160 << 20,), dtype=torch.float32, device="cuda")  # 640 MB, more than L2

    def chain(flags, evict=False):
        for t in mid + mid_l + fin + fin_l:
            t.fill_(float("nan"))
        if evict:  # the NaN lines go back to DRAM, so B's prefetch brings them from there
            flush.add_(1.0)
        dcp.merge(srcs, lses, False, outs=mid, lse_outs=mid_l, flags=flags)
        dcp.merge(mid, mid_l, False, outs=fin, lse_outs=fin_l, flags=flags)
        torch.cuda.synchronize()
        return _bits(mid) + _bits(mid_l) + _bits(fin) + _bits(fin_l)

    ref = chain(0)
    assert not any(bool(torch.isnan(t).any()) for t in fin)
    for it in range(20):
        flags = dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH | (dcp.DCP_FLAG_LSE_FIRST if it % 2 else 0)
        assert all(torch.equal(a, b) for a, b in zip(ref, chain(flags, evict=it % 4 < 2))), f"iteration {it}"


@pytest.mark.parametrize("flags", [dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH,
                                   dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH | dcp.DCP_FLAG_LSE_FIRST,
                                   dcp.DCP_FLAG_PREFETCH | dcp.DCP_FLAG_PRELOAD])
@pytest.mark.parametrize("cfg,rows", [("kimi", 1), ("kimi", 128), ("kimi", 512), ("deepseek", 64)])
def test_prefetch_flags_match_the_oracle(oracle_mod, flags, cfg, rows):
    check_against_oracle(oracle_mod, make_merge_inputs(cfg, rows, seed=7), flags=flags, what=f"{cfg} B={rows}")


@pytest.mark.parametrize("pdl", [False, True])
def test_graph_replay_is_bit_identical_and_interleaves_with_eager(pdl):
    inp = make_merge_inputs("kimi", 16, seed=3)
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    outs = [torch.empty((16, 16, 512), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    louts = [torch.empty((16, 16), dtype=torch.float32, device="cuda") for _ in range(4)]
    flags = dcp.DCP_FLAG_PDL if pdl else 0
    eager_o, eager_l = dcp.merge(srcs, lses, False, flags=flags)
    ref = _bits(eager_o) + _bits(eager_l)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dcp.merge(srcs, lses, False, outs=outs, lse_outs=louts, flags=flags)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(10):
            dcp.merge(srcs, lses, False, outs=outs, lse_outs=louts, flags=flags)
    for it in range(5):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(ref, _bits(outs) + _bits(louts))), f"replay {it}"
        # eager call between replays, on other outputs
        o2, l2 = dcp.merge(srcs, lses, False, flags=flags)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(ref, _bits(o2) + _bits(l2)))


def test_graph_replay_sees_changed_inputs(oracle_mod):
    # a captured call reads its buffers at replay time
    a = make_merge_inputs("kimi", 8, seed=10)
    b = make_merge_inputs("kimi", 8, seed=11)
    srcs = [to_dev_bits(s) for s in a.srcs]
    lses = [torch.from_numpy(l).cuda() for l in a.lses]
    outs = [torch.empty((8, 16, 512), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    louts = [torch.empty((8, 16), dtype=torch.float32, device="cuda") for _ in range(4)]
    dcp.merge(srcs, lses, False, outs=outs, lse_outs=louts)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dcp.merge(srcs, lses, False, outs=outs, lse_outs=louts)
    for j in range(4):
        srcs[j].copy_(to_dev_bits(b.srcs[j]))
        lses[j].copy_(torch.from_numpy(b.lses[j]).cuda())
    g.replay()
    torch.cuda.synchronize()
    ref, lref = oracle_mod.merge(b.srcs, b.lses, False)
    for r in range(4):
        assert_out_close(outs[r].float().double().cpu().numpy(), ref[r], "replay with new inputs")
        assert_lse_close(louts[r].double().cpu().numpy(), lref[r])


def test_runs_on_a_side_stream_in_order():
    inp = make_merge_inputs("kimi", 32, seed=12)
    srcs = [to_dev_bits(s) for s in inp.srcs]
    lses = [torch.from_numpy(l).cuda() for l in inp.lses]
    ref_o, _ = dcp.merge(srcs, lses, False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            o, _ = dcp.merge(srcs, lses, False, flags=dcp.DCP_FLAG_PDL)
    s.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(_bits(ref_o), _bits(o)))


def test_batch_beyond_one_launch_is_split_and_exact():
    """The largest batch the merge takes in one launch is 2^30 (row, head)
    units; a larger one runs as several launches over row ranges. Here cp = 2,
    H = 16 (8 per destination), D = 8 and 2^26 + 3 rows: 2^30 + 48 units, two
    launches, about 60 GiB of buffers. Both sources have the same LSE, so each
    weight is exactly 1/2 and the output is the bf16 rounding of the exact
    mean, the merged LSE lse + ln 2 in fp32; checked bit for bit everywhere,
    on the device, in row chunks."""
    free, _ = torch.cuda.mem_get_info()
    if free < (72 << 30):
        pytest.skip("needs about 60 GiB of free device memory")
    cp, H, D = 2, 16, 8
    Hl = H // cp
    B = (1 << 26) + 3
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    chunk = 1 << 22
    srcs = [torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    for b0 in range(0, B, chunk):
        b1 = min(B, b0 + chunk)
        for s in srcs:
            s[b0:b1] = torch.randn((b1 - b0, H, D), generator=gen, device="cuda").to(torch.bfloat16)
        lse[b0:b1] = torch.randn((b1 - b0, H), generator=gen, device="cuda") * 6.0 + 10.0
    lses = [lse, lse.clone()]
    outs, louts = dcp.merge(srcs, lses, True)
    torch.cuda.synchronize()
    ln2 = torch.tensor(0.6931471805599453, dtype=torch.float32, device="cuda")
    for b0 in range(0, B, chunk):
        b1 = min(B, b0 + chunk)
        for r in range(cp):
            h = slice(r * Hl, (r + 1) * Hl)
            want = ((srcs[0][b0:b1, h].float() + srcs[1][b0:b1, h].float()) * 0.5).to(torch.bfloat16)
            assert torch.equal(outs[r][b0:b1].view(torch.int16), want.view(torch.int16)), f"rows {b0}.. dest {r}"
            want_l = lse[b0:b1, h] + ln2
            assert torch.equal(louts[r][b0:b1].view(torch.int32), want_l.view(torch.int32)), f"LSE rows {b0}.. {r}"
