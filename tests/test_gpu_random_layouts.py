"""Seeded random cases of the strided merge (dcp_lse_reduce_ex) against the
oracle: every generality feature at once, in combinations the targeted tests
do not reach. Per case: cp in 1..16, 1..4 heads per destination, D from 8 to
520, bf16 or fp16, base 2 or e, padded source / LSE / destination strides, an
LSE head stride of 1..3 (FlashMLA's [B, H, s_q] layout), a launch flag set
(schedules, PDL, the L2 prefetch), empty shards (LSE -inf, payload NaN) or
seq_lens masking (LSE NaN, payload NaN). Padding in the inputs holds NaN and
must never be read; padding in the outputs holds a sentinel and must never
be written."""
import numpy as np
import pytest
import torch

import decode_context_mla_dcp_gb300 as dcp
from decode_context_mla_dcp_gb300 import build as dcp_build
from decode_context_mla_dcp_gb300.inputs import BF16_QNAN, F16_QNAN, bf16_bits, f16_bits

pytestmark = pytest.mark.gpu

FLAG_SETS = [0, dcp.DCP_FLAG_PDL, dcp.DCP_FLAG_PRELOAD, dcp.DCP_FLAG_LSE_FIRST,
             dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH, dcp.DCP_FLAG_PREFETCH | dcp.DCP_FLAG_LSE_FIRST,
             dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PRELOAD | dcp.DCP_FLAG_PREFETCH]
OUT_SENTINEL = 0x7E01
LSE_SENTINEL = 0x7FBADBAD


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    dcp_build.build()
    dcp.load()
    torch.cuda.set_device(0)
    yield


def draw_case(case: int):
    rng = np.random.default_rng([2024, case])
    c = {}
    c["cp"] = cp = int(rng.integers(1, 17))
    c["Hl"] = Hl = int(rng.integers(1, 5))
    c["H"] = H = cp * Hl
    c["D"] = D = int(rng.choice([8, 16, 64, 136, 512, 520]))
    c["B"] = B = int(rng.integers(1, 33))
    c["dtype"] = "f16" if rng.random() < 0.3 else "bf16"
    c["base_e"] = bool(rng.integers(0, 2))
    c["src_head"] = D + 8 * int(rng.integers(0, 3))
    c["src_row"] = H * c["src_head"] + 8 * int(rng.integers(0, 4))
    c["lse_head"] = int(rng.integers(1, 4))
    c["lse_row"] = H * c["lse_head"] + int(rng.integers(0, 5))
    c["dst_head"] = D + 8 * int(rng.integers(0, 3))
    c["dst_row"] = Hl * c["dst_head"] + 8 * int(rng.integers(0, 3))
    c["lse_out_row"] = Hl + int(rng.integers(0, 3))
    c["flags"] = FLAG_SETS[int(rng.integers(len(FLAG_SETS)))]
    mode = rng.choice(["plain", "empty", "seq_lens"], p=[0.4, 0.3, 0.3])
    c["mode"] = str(mode)
    c["interleave"] = int(rng.choice([1, 2, 16]))

    to_bits = bf16_bits if c["dtype"] == "bf16" else f16_bits
    qnan = BF16_QNAN if c["dtype"] == "bf16" else F16_QNAN
    payload = [to_bits(rng.standard_normal((B, H, D), dtype=np.float32)) for _ in range(cp)]
    if c["base_e"]:
        lse = [rng.normal(10.0, 6.0, size=(B, H)).astype(np.float32) for _ in range(cp)]
    else:
        lse = [rng.uniform(-4.0, 24.0, size=(B, H)).astype(np.float32) for _ in range(cp)]
    lens = None
    if mode == "empty":
        empty = rng.random((B, cp)) < 0.25
        for j in range(cp):
            lse[j][empty[:, j]] = -np.inf
            payload[j][empty[:, j]] = qnan
    elif mode == "seq_lens":
        lens = rng.integers(0, cp * c["interleave"] + 3, size=B).astype(np.int32)
        for j in range(cp):
            empty = lens <= j * c["interleave"]
            lse[j][empty] = np.nan
            payload[j][empty] = qnan
    c["lens"] = lens

    # backing arrays with NaN padding
    bi = np.arange(B)[:, None] * c["src_row"] + np.arange(H)[None, :] * c["src_head"]
    li = np.arange(B)[:, None] * c["lse_row"] + np.arange(H)[None, :] * c["lse_head"]
    c["src_back"], c["lse_back"] = [], []
    for j in range(cp):
        s = np.full(B * c["src_row"], qnan, dtype=np.uint16)
        s[bi[..., None] + np.arange(D)] = payload[j]
        c["src_back"].append(s.reshape(B, c["src_row"]))
        l = np.full(B * c["lse_row"], np.nan, dtype=np.float32)
        l[li] = lse[j]
        c["lse_back"].append(l.reshape(B, c["lse_row"]))
    return c


@pytest.mark.parametrize("case", range(48))
def test_random_strided_merges_match_the_oracle(oracle_mod, case):
    c = draw_case(case)
    cp, B, H, Hl, D = c["cp"], c["B"], c["H"], c["Hl"], c["D"]
    tdt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float16
    srcs = [torch.from_numpy(s.view(np.int16)).view(tdt).cuda() for s in c["src_back"]]
    lses = [torch.from_numpy(l).cuda() for l in c["lse_back"]]
    dsts = [torch.full((B * c["dst_row"],), OUT_SENTINEL, dtype=torch.int32, device="cuda").to(torch.int16)
            for _ in range(cp)]
    louts = [torch.full((B * c["lse_out_row"],), LSE_SENTINEL, dtype=torch.int32, device="cuda")
             for _ in range(cp)]
    seq = torch.from_numpy(c["lens"]).cuda() if c["lens"] is not None else None
    layout = dcp.Layout(src_row=c["src_row"], src_head=c["src_head"], lse_row=c["lse_row"], lse_head=c["lse_head"],
                        dst_row=c["dst_row"], dst_head=c["dst_head"], lse_out_row=c["lse_out_row"])
    dcp.dcp_lse_reduce_ex(srcs, lses, cp, B, H, D, c["base_e"],
                          dcp.DCP_DTYPE_BF16 if c["dtype"] == "bf16" else dcp.DCP_DTYPE_F16, dsts, louts,
                          layout=layout, flags=c["flags"], seq_lens=seq, interleave=c["interleave"])
    torch.cuda.synchronize()

    ref, lref = oracle_mod.merge(c["src_back"], c["lse_back"], c["base_e"], dtype=c["dtype"], H=H, D=D,
                                 src_strides=(c["src_row"], c["src_head"]),
                                 lse_strides=(c["lse_row"], c["lse_head"]), seq_lens=c["lens"],
                                 interleave=c["interleave"])
    what = {k: v for k, v in c.items() if k not in ("src_back", "lse_back", "lens")}
    oi = np.arange(B)[:, None] * c["dst_row"] + np.arange(Hl)[None, :] * c["dst_head"]
    loi = np.arange(B)[:, None] * c["lse_out_row"] + np.arange(Hl)[None, :]
    for r in range(cp):
        back = dsts[r].cpu().numpy().view(np.uint16)
        bits = back[oi[..., None] + np.arange(D)]
        if c["dtype"] == "bf16":
            got = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            tight = 2.0 ** -8 * np.abs(ref[r]) + 1e-5
        else:
            got = bits.view(np.float16).astype(np.float64)
            tight = 2.0 ** -11 * np.abs(ref[r]) + 1e-5
        assert not np.isnan(got).any(), f"NaN output, {what}"
        err = np.abs(got - ref[r])
        assert (err <= 1e-2 + 8e-3 * np.abs(ref[r])).all() and (err <= tight).all(), \
            f"dest {r}: max err {err.max():.3g}, {what}"
        mask = np.ones(back.size, dtype=bool)
        mask[(oi[..., None] + np.arange(D)).ravel()] = False
        assert (back[mask] == OUT_SENTINEL).all(), f"a write outside dest {r}'s elements, {what}"

        lback = louts[r].cpu().numpy()
        got_l = lback[loi].view(np.float32).astype(np.float64)
        fin = np.isfinite(lref[r])
        assert np.array_equal(np.isfinite(got_l), fin) and not np.isnan(got_l).any(), f"LSE pattern, {what}"
        lerr = np.abs(got_l[fin] - lref[r][fin])
        assert (lerr <= 1e-5 * np.maximum(np.abs(lref[r][fin]), 1.0)).all(), f"LSE dest {r}, {what}"
        lmask = np.ones(lback.size, dtype=bool)
        lmask[loi.ravel()] = False
        assert (lback[lmask].view(np.uint32) == LSE_SENTINEL).all(), f"a write outside lse_out {r}, {what}"
