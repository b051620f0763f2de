"""Host-side checks of the C ABI: the library builds, loads and exports every
function include/dcp_lse_reduce.h declares, and bad arguments are rejected on
the host with the documented status (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

import decode_context_mla_dcp_gb300 as dcp
from decode_context_mla_dcp_gb300 import build as dcp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    dcp_build.build()
    return dcp.load()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dcp_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_exported_api():
    assert declared_functions() == sorted(dcp.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_messages(lib):
    assert dcp.dcp_lse_reduce_version() == 10000
    assert "multiple of cp" in dcp.dcp_lse_reduce_strerror(-4)
    assert dcp.dcp_lse_reduce_strerror(0) == "success"


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced on the host


def call(lib, cp=2, B=1, H=4, D=512, lse_stride=None, srcs=None, lses=None, dsts=None, lse_outs=None,
         base_e=1):
    arr = ctypes.c_void_p * max(cp, 1)
    srcs = arr(*([FAKE] * max(cp, 1))) if srcs is None else srcs
    lses = arr(*([FAKE] * max(cp, 1))) if lses is None else lses
    dsts = arr(*([FAKE + 4096] * max(cp, 1))) if dsts is None else dsts
    return lib.dcp_lse_reduce(srcs, lses, H if lse_stride is None else lse_stride, cp, B, H, D, base_e,
                              dsts, lse_outs, None)


@pytest.mark.parametrize("kw,status", [
    (dict(cp=0), -2), (dict(cp=17, H=17), -2), (dict(B=-1), -3), (dict(H=0), -3),
    (dict(D=0), -3), (dict(D=12), -3), (dict(H=6, cp=4), -4), (dict(lse_stride=3), -5),
])
def test_bad_arguments_are_rejected(lib, kw, status):
    assert call(lib, **kw) == status


def test_null_pointers_are_rejected(lib):
    arr = ctypes.c_void_p * 2
    assert lib.dcp_lse_reduce(None, arr(FAKE, FAKE), 4, 2, 1, 4, 512, 1, arr(FAKE, FAKE), None, None) == -1
    assert call(lib, srcs=arr(FAKE, 0)) == -1
    assert call(lib, dsts=arr(0, FAKE)) == -1


def test_misaligned_pointers_are_rejected(lib):
    arr = ctypes.c_void_p * 2
    assert call(lib, srcs=arr(FAKE, FAKE + 8)) == -6
    assert call(lib, dsts=arr(FAKE + 2, FAKE)) == -6
    assert call(lib, lses=arr(FAKE + 2, FAKE)) == -6
    assert call(lib, lse_outs=arr(FAKE + 1, 0)) == -6


def test_empty_batch_is_a_no_op(lib):
    # B = 0 returns before touching the device
    assert call(lib, B=0) == 0


def test_ex_rejects_bad_flags_dtype_strides(lib):
    arr = ctypes.c_void_p * 2
    p = arr(FAKE, FAKE)
    q = arr(FAKE + 4096, FAKE + 4096)

    def ex(dtype=0, flags=0, layout=None, base_e=1, seq_lens=None, interleave=1):
        return lib.dcp_lse_reduce_ex(p, p, 2, 1, 4, 512, base_e, dtype, q, None,
                                     ctypes.byref(layout) if layout is not None else None, seq_lens, interleave,
                                     flags, None)

    assert ex(dtype=2) == -8
    assert ex(base_e=2) == -9
    assert ex(flags=32) == -7
    assert ex(flags=dcp.DCP_FLAG_PRELOAD | dcp.DCP_FLAG_LSE_FIRST) == -7
    assert ex(flags=16) == -7
    assert ex(flags=dcp.DCP_FLAG_PRELOAD | dcp.DCP_FLAG_LSE_FIRST | dcp.DCP_FLAG_PREFETCH) == -7
    assert ex(seq_lens=FAKE, interleave=0) == -11
    assert ex(seq_lens=FAKE, interleave=(1 << 24) + 1) == -11
    assert ex(seq_lens=FAKE + 2, interleave=1) == -6
    good = dict(src_row=2048, src_head=512, lse_row=4, lse_head=1, dst_row=1024, dst_head=512, lse_out_row=2)
    for key, bad in [("src_row", 2044), ("src_head", 4), ("dst_row", -8), ("dst_head", 12), ("lse_row", -1)]:
        lay = dcp.Layout(**{**good, key: bad})
        assert ex(layout=lay) == -5, key


def test_python_binding_raises_with_message(lib):
    with pytest.raises(dcp.DcpError, match="multiple of cp"):
        dcp.dcp_lse_reduce([FAKE] * 4, [FAKE] * 4, 6, 4, 1, 6, 512, True, [FAKE] * 4, stream=0)


def test_mla_producer_rejects_bad_arguments(lib):
    arr = ctypes.c_void_p * 2
    outs = arr(FAKE, FAKE)
    lses = arr(FAKE, FAKE)

    def call(q=FAKE, kv=FAKE, kv_len=FAKE, B=1, H=64, Dk=576, Dv=512, T=10, n_split=2, o=outs, l=lses, status=None,
             flags=0):
        return lib.dcp_mla_decode_partial(q, kv, kv_len, B, H, Dk, Dv, T, 0.1, 1, n_split, o, l, status, flags,
                                          None)

    assert call(q=None) == -101
    assert call(o=arr(FAKE, 0)) == -101
    assert call(B=-1) == -102 and call(B=65536) == -102
    assert call(H=8) == -102 and call(H=24) == -102
    assert call(Dk=640) == -102 and call(Dv=256) == -102 and call(T=-1) == -102
    assert call(n_split=0) == -103 and call(n_split=17) == -103
    assert call(q=FAKE + 8) == -104 and call(kv_len=FAKE + 2) == -104 and call(o=arr(FAKE + 4, FAKE)) == -104
    assert call(flags=16) == -105 and call(flags=6) == -105  # the one-kernel flag is dcp_mla_decode's only
    assert call(flags=64) == -105
    assert call(flags=dcp.DCP_MLA_FLAG_TEST_STALL | dcp.DCP_MLA_FLAG_MMA_SYNC, B=0) == 0  # the stall test is known
    assert call(flags=dcp.DCP_FLAG_PREFETCH | dcp.DCP_FLAG_PDL, B=0) == 0  # the producer takes the prefetch flag
    assert call(B=0) == 0  # nothing to do, nothing launched
    assert dcp.dcp_mla_decode_smem_bytes(576, 64) > 150000
    assert "n_split" in dcp.dcp_lse_reduce_strerror(-103)


def test_every_status_code_has_a_message_in_the_c_library(lib):
    # The producer's and the fused decode's codes are explained by the C
    # library itself, so a C caller needs no table of its own.
    lib.dcp_lse_reduce_strerror.restype = ctypes.c_char_p
    assert b"n_split" in lib.dcp_lse_reduce_strerror(-103)
    for code in list(range(-11, 0)) + list(range(-110, -100)):
        msg = lib.dcp_lse_reduce_strerror(code)
        assert msg and msg != b"unknown status", code
    assert lib.dcp_lse_reduce_strerror(-12) == b"unknown status"
    assert lib.dcp_lse_reduce_strerror(-100) == b"unknown status"


def test_fused_decode_rejects_bad_workspace_and_cp(lib):
    need = dcp.dcp_mla_decode_workspace_bytes(4, 2, 3, 64)
    assert need == 8 * (3 * 64 * 512 * 2 + 768)  # both parts are already multiples of 256 bytes
    arr = ctypes.c_void_p * 4
    kv = arr(FAKE, FAKE, FAKE, FAKE)
    lens = arr(FAKE, FAKE, FAKE, FAKE)
    dst = arr(FAKE, FAKE, FAKE, FAKE)

    def call(cp=4, n_split=2, H=64, ws=FAKE, ws_bytes=None):
        return lib.dcp_mla_decode(FAKE, kv, lens, cp, 3, H, 576, 512, 100, 0.1, 1, n_split, ws,
                                  need if ws_bytes is None else ws_bytes, dst, None, None, 0, None)

    assert call(ws_bytes=need - 1) == -106
    assert call(ws=FAKE + 128) == -106
    assert call(ws=None) == -106
    assert call(n_split=8) == -107          # 4 * 8 sources > 16
    assert call(n_split=3) == -107          # 64 % 12 != 0
    assert call(H=36) == -102               # not a multiple of 16: a shape error, reported first
    assert call(cp=0) == -107


def test_producer_kernel_choice(lib):
    """The producer's default kernel by head block and split length, the
    forcing flags, and rejected arguments (host only)."""
    tc, mma = dcp.DCP_MLA_KERNEL_TCGEN05, dcp.DCP_MLA_KERNEL_MMA_SYNC
    k = dcp.dcp_mla_decode_kernel
    # 64-head blocks: tcgen05 from one full 128-token tile per split
    assert k(128, 4096, 9) == tc and k(64, 4096, 16) == tc and k(64, 2048, 16) == tc
    assert k(64, 2032, 16) == mma and k(128, 100, 1) == mma  # ceil(2032 / 16) = 127 tokens per split
    # 32-head blocks: from two tiles
    assert k(32, 2048, 8) == tc and k(96, 2048, 8) == tc and k(32, 2040, 8) == mma and k(32, 1024, 8) == mma
    # 16-head blocks: always mma.sync by default
    assert k(16, 1 << 20, 1) == mma and k(48, 1 << 20, 1) == mma
    # forcing flags (PDL does not change the choice)
    assert k(16, 64, 1, dcp.DCP_MLA_FLAG_TCGEN05) == tc and k(128, 1 << 20, 1, dcp.DCP_MLA_FLAG_MMA_SYNC) == mma
    assert k(128, 4096, 1, dcp.DCP_FLAG_PDL) == tc and k(128, 4096, 1, dcp.DCP_FLAG_PREFETCH) == tc
    assert k(128, 4096, 1, dcp.DCP_MLA_FLAG_TEST_STALL) == tc and k(16, 64, 1, dcp.DCP_MLA_FLAG_TEST_STALL) == mma
    for args, status in [((128, 4096, 1, dcp.DCP_MLA_FLAG_TCGEN05 | dcp.DCP_MLA_FLAG_MMA_SYNC), -105),
                         ((128, 4096, 1, 16), -105), ((128, 4096, 0), -103), ((128, 4096, 17), -103),
                         ((20, 4096, 1), -102), ((128, -1, 1), -102)]:
        with pytest.raises(dcp.DcpError) as e:
            k(*args)
        assert e.value.status == status
    # the shared-memory query covers the larger (tcgen05) kernel
    assert dcp.dcp_mla_decode_smem_bytes(576, 64) == 224256  # 144 KB tile + 72 KB Q + misc + alignment
    assert dcp.dcp_mla_decode_smem_bytes(500, 64) == -1 and dcp.dcp_mla_decode_smem_bytes(576, 20) == -1


def test_split_count_pick(lib):
    """One wave of CTAs, at least one 128-token tile per split, H a multiple
    of cp*n_split, cp*n_split <= 16 (host only)."""
    pick = dcp.dcp_mla_decode_pick_split
    # DeepSeek-like fused decode: 8 shards x 2 head blocks x 8 rows = 128 CTAs per split count
    assert pick(8, 8, 128, 512, 152) == 1
    # Kimi-like: 4 shards x 1 head block x 8 rows = 32 CTAs per split count -> 4 (128 CTAs; 16 / cp = 4)
    assert pick(4, 8, 64, 1024, 152) == 4
    # one shard, 8 rows x 2 blocks = 16 CTAs per split: 9 fit a wave but 128 % 9 != 0 -> 8
    assert pick(1, 8, 128, 4096, 152) == 8
    # short caches cap the split count at one tile per split
    assert pick(1, 1, 128, 300, 152) == 2 and pick(1, 1, 128, 100, 152) == 1
    # a batch that already fills the GPU gets one split
    assert pick(1, 200, 64, 1 << 16, 152) == 1
    # 16-head blocks run on the mma.sync kernel, two CTAs per SM: a wave holds 304 of them
    assert pick(1, 148, 16, 4096, 152) == 2 and pick(1, 64, 16, 2048, 152) == 4
    # every pick is a valid producer / fused split count
    for cp, B, H, T in [(1, 1, 16, 1 << 16), (2, 3, 96, 5000), (8, 1, 128, 32768), (16, 1, 256, 1 << 20)]:
        n = pick(cp, B, H, T, 152)
        assert 1 <= n and cp * n <= 16 and H % (cp * n) == 0
    for args, status in [((0, 8, 128, 512, 152), -107), ((3, 8, 128, 512, 152), -107), ((17, 8, 272, 512, 152), -107),
                         ((1, 8, 20, 512, 152), -102), ((1, -1, 128, 512, 152), -102), ((1, 8, 128, 512, 0), -102)]:
        with pytest.raises(dcp.DcpError) as e:
            pick(*args)
        assert e.value.status == status


def test_no_alloc_reports_bad_shapes_before_the_scratch_limit(lib):
    # A shape the producer rejects is a shape error even when its partials
    # would not fit the built-in scratch array; checked on the host, nothing
    # launched, no device needed.
    arr = ctypes.c_void_p * 8
    ptrs = arr(*[FAKE] * 8)

    def noalloc(B=64, H=128, Dk=576, Dv=512, T=100, cp=8, n_split=2):
        return lib.dcp_mla_decode_noalloc(FAKE, ptrs, ptrs, cp, B, H, Dk, Dv, T, 0.1, 1, n_split, ptrs, None, None,
                                          0, None)

    def fused(B=64, H=128, Dk=576, Dv=512, T=100, cp=8, n_split=2, ws_bytes=1 << 20):
        return lib.dcp_mla_decode(FAKE, ptrs, ptrs, cp, B, H, Dk, Dv, T, 0.1, 1, n_split, FAKE, ws_bytes, ptrs, None,
                                  None, 0, None)

    assert noalloc() == -108                      # valid shape, too large for the scratch
    assert noalloc(Dv=4096) == -102 and noalloc(B=70000) == -102 and noalloc(Dk=640) == -102
    assert noalloc(H=8, cp=1, n_split=1) == -102  # H not a multiple of 16
    assert noalloc(n_split=17) == -103 and noalloc(cp=16) == -107
    assert fused(Dv=4096) == -102 and fused(B=-1) == -102
    assert fused() == -106                        # valid shape, workspace too small
    need = dcp.dcp_mla_decode_workspace_bytes(8, 2, 0, 128)
    assert fused(B=0, ws_bytes=1 << 20, ) == 0 and need == 0
    assert lib.dcp_mla_decode(FAKE, ptrs, ptrs, 8, 0, 128, 576, 512, 100, 0.1, 1, 2, FAKE, 1 << 20, ptrs, None, None,
                              dcp.DCP_MLA_FLAG_ONE_KERNEL | dcp.DCP_FLAG_PDL, None) == 0
    assert lib.dcp_mla_decode(FAKE, ptrs, ptrs, 8, 0, 128, 576, 512, 100, 0.1, 1, 2, FAKE, 1 << 20, ptrs, None, None,
                              64, None) == -105
