"""Pins for the CPU oracle: facts fixed by the mathematics of the merge, not by
the oracle's own code.

The merge (named on "[DCP] Run fi_a2a on FlashInfer's fused all-to-all + LSE
reduce", "Motivation", and "[Attention] Add direct symmetric-memory DCP A2A",
commit notes: FP32 LSE weighting, base 2 or e) is the split-softmax merge. Each
test below would fail on a plausible slip in the oracle:

* dropped normalisation           -> equal-LSE mean, hand-worked case
* exponent sign flipped           -> hand-worked case
* no max shift (overflow)         -> shift invariance at +-1000
* base-2 treated as base e        -> hand-worked base-2 case, base agreement
* wrong merged-LSE formula        -> equal-LSE LSE, full-attention LSE
* head routed to h % cp           -> one-hot head routing
* stride misuse / reads padding   -> LSE stride padding with NaN
* -inf source weighted or read    -> NaN-payload shard, empty row
"""
import math

import numpy as np
import pytest

from decode_context_mla_dcp_gb300.inputs import bf16_bits, make_merge_inputs, tiny_qkv

LN2 = math.log(2.0)


def concat_heads(outs):
    """Destinations r = 0..cp-1 own consecutive head blocks: concatenating them
    along the head axis gives the merge for every head, [B, H, D]."""
    return np.concatenate(outs, axis=1)


def widen_bf16(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --- 16-bit widening ------------------------------------------------------

@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x3F81, 1.0 + 2.0 ** -7), (0x4049, 3.140625),
    (0x0001, 2.0 ** -133), (0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127), (0x8000, -0.0),
    (0x7F80, math.inf), (0xFF80, -math.inf)])
def test_bf16_widening_textbook_values(oracle_mod, bits, value):
    assert oracle_mod.half_bits_to_double("bf16", bits) == value


def test_bf16_widening_nan(oracle_mod):
    assert math.isnan(oracle_mod.half_bits_to_double("bf16", 0x7FC0))


def test_f16_widening_matches_numpy_for_every_pattern(oracle_mod):
    ref = np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_bits_to_double("f16", b) for b in range(1 << 16)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


# --- closed forms ---------------------------------------------------------

@pytest.mark.parametrize("base_e", [True, False])
def test_cp1_is_identity(oracle_mod, base_e):
    inp = make_merge_inputs("kimi", rows=5, seed=3, cp=1, H=8, D=64)
    outs, lse_outs = oracle_mod.merge(inp.srcs, inp.lses, base_e)
    assert np.array_equal(outs[0], widen_bf16(inp.srcs[0]))
    np.testing.assert_allclose(lse_outs[0], inp.lses[0].astype(np.float64), rtol=1e-15, atol=0)


@pytest.mark.parametrize("cp", [2, 4, 8])
@pytest.mark.parametrize("base_e", [True, False])
def test_equal_lse_gives_exact_mean(oracle_mod, cp, base_e):
    inp = make_merge_inputs("kimi", rows=3, seed=5, cp=cp, H=2 * cp, D=32)
    lse = np.full((3, 2 * cp), 7.25, dtype=np.float32)
    outs, lse_outs = oracle_mod.merge(inp.srcs, [lse] * cp, base_e)
    mean = sum(widen_bf16(s) for s in inp.srcs) / cp
    np.testing.assert_allclose(concat_heads(outs), mean, rtol=1e-14, atol=1e-15)
    # log_b(cp * b^7.25) = 7.25 + log_b(cp)
    expect = 7.25 + (math.log(cp) if base_e else math.log2(cp))
    np.testing.assert_allclose(concat_heads([l[..., None] for l in lse_outs])[..., 0], expect, rtol=1e-15)


def _hand_case(base_e):
    # cp = 4 sources, one head, one row, D = 4. Base-2 LSEs [2, 0, 0, 1] give
    # unnormalised weights 4, 1, 1, 2 (sum 8), i.e. 1/2, 1/8, 1/8, 1/4, and a
    # merged LSE of log2(8) = 3. Per-feature payloads (bf16-exact):
    #   d=0: 1, -2, 0.5, 4   -> 0.5 - 0.25 + 0.0625 + 1    = 1.3125
    #   d=1: 8, 8, 8, 8      -> 8
    #   d=2: 0, 16, 0, 0     -> 2
    #   d=3: -1, 0, 0, 1     -> -0.5 + 0.25               = -0.25
    # One head per destination needs H = cp = 4; heads other than 0 copy the
    # same values, so every destination sees the same case.
    payload = np.array([[1, 8, 0, -1], [-2, 8, 16, 0], [0.5, 8, 0, 0], [4, 8, 0, 1]], dtype=np.float32)
    srcs = [np.broadcast_to(bf16_bits(payload[j]), (1, 4, 4)).copy() for j in range(4)]
    lse2 = np.array([2.0, 0.0, 0.0, 1.0])
    lse = lse2 * LN2 if base_e else lse2
    lses = [np.full((1, 4), lse[j], dtype=np.float64) for j in range(4)]
    return srcs, lses


@pytest.mark.parametrize("base_e", [False, True])
def test_hand_worked_dyadic_case(oracle_mod, base_e):
    srcs, lses = _hand_case(base_e)
    outs, lse_outs = oracle_mod.merge(srcs, lses, base_e)
    expect = np.array([1.3125, 8.0, 2.0, -0.25])
    expect_lse = 3.0 * LN2 if base_e else 3.0
    for r in range(4):
        np.testing.assert_allclose(outs[r][0, 0], expect, rtol=1e-15, atol=1e-15)
        assert abs(lse_outs[r][0, 0] - expect_lse) <= 1e-15 * 4


def test_neg_inf_source_has_zero_weight_even_with_nan_payload(oracle_mod):
    inp = make_merge_inputs("deepseek", rows=4, seed=7, cp=3, H=6, D=16)
    lses = [l.reshape(4, 6).copy() for l in inp.lses]
    lses[1][:] = -np.inf
    nan_srcs = list(inp.srcs)
    nan_srcs[1] = np.full_like(inp.srcs[1], 0x7FC0)
    a, la = oracle_mod.merge(nan_srcs, lses, True)
    # same merge with a finite payload behind the -inf LSE
    b, lb = oracle_mod.merge(inp.srcs, lses, True)
    # and with the source pushed so far down that exp underflows to exactly 0
    lses_far = [l.astype(np.float64) for l in lses]
    lses_far[1] = np.minimum(lses_far[0], lses_far[2]) - 2000.0
    c, lc = oracle_mod.merge(inp.srcs, lses_far, True)
    for r in range(3):
        assert np.isfinite(a[r]).all()
        assert np.array_equal(a[r], b[r]) and np.array_equal(a[r], c[r])
        assert np.array_equal(la[r], lb[r]) and np.array_equal(la[r], lc[r])


def test_row_with_every_source_empty(oracle_mod):
    inp = make_merge_inputs("kimi", rows=3, seed=1, cp=4, H=8, D=16)
    lses = [l.copy() for l in inp.lses]
    srcs = [s.copy() for s in inp.srcs]
    for j in range(4):
        lses[j][1] = -np.inf
        srcs[j][1] = 0x7FC0
    outs, lse_outs = oracle_mod.merge(srcs, lses, False)
    for r in range(4):
        assert np.array_equal(outs[r][1], np.zeros_like(outs[r][1]))
        assert np.all(lse_outs[r][1] == -np.inf)
        assert np.isfinite(outs[r][[0, 2]]).all() and np.isfinite(lse_outs[r][[0, 2]]).all()


def test_base2_and_base_e_agree(oracle_mod):
    inp = make_merge_inputs("deepseek", rows=5, seed=11, cp=4, H=8, D=32)
    lse_e = [l.reshape(5, 8).astype(np.float64) for l in inp.lses]
    lse_2 = [l / LN2 for l in lse_e]
    oe, le = oracle_mod.merge(inp.srcs, lse_e, True)
    o2, l2 = oracle_mod.merge(inp.srcs, lse_2, False)
    for r in range(4):
        np.testing.assert_allclose(o2[r], oe[r], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(l2[r] * LN2, le[r], rtol=1e-13)


@pytest.mark.parametrize("shift", [1000.0, -1000.0, 0.5])
def test_shift_invariance(oracle_mod, shift):
    inp = make_merge_inputs("kimi", rows=4, seed=13, cp=4, H=8, D=16)
    base = [l.astype(np.float64) for l in inp.lses]
    o0, l0 = oracle_mod.merge(inp.srcs, base, True)
    o1, l1 = oracle_mod.merge(inp.srcs, [l + shift for l in base], True)
    for r in range(4):
        assert np.isfinite(o1[r]).all()
        np.testing.assert_allclose(o1[r], o0[r], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(l1[r], l0[r] + shift, rtol=1e-13, atol=1e-10)


def test_nested_merges_are_associative(oracle_mod):
    # Merging shards {0,1} and {2,3} first, then merging the two results,
    # equals merging all four at once (what lets DCP split a context anywhere).
    rng = np.random.default_rng(17)
    B, H, D = 3, 8, 24
    srcs = [rng.standard_normal((B, H, D)) for _ in range(4)]
    lses = [rng.normal(3.0, 2.0, (B, H)) for _ in range(4)]
    o_all, l_all = oracle_mod.merge(srcs, lses, True, dtype="f64")
    o01, l01 = oracle_mod.merge(srcs[:2], lses[:2], True, dtype="f64")
    o23, l23 = oracle_mod.merge(srcs[2:], lses[2:], True, dtype="f64")
    pair_srcs = [concat_heads(o01), concat_heads(o23)]
    pair_lses = [np.concatenate(l01, axis=1), np.concatenate(l23, axis=1)]
    o_pair, l_pair = oracle_mod.merge(pair_srcs, pair_lses, True, dtype="f64")
    np.testing.assert_allclose(concat_heads(o_pair), concat_heads(o_all), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(np.concatenate(l_pair, 1), np.concatenate(l_all, 1), rtol=1e-13)


def test_convex_combination(oracle_mod):
    inp = make_merge_inputs("stress", rows=6, seed=19, cp=8, H=16, D=64)
    outs, _ = oracle_mod.merge(inp.srcs, inp.lses, True)
    x = np.stack([widen_bf16(s) for s in inp.srcs])       # [cp, B, H, D]
    got = concat_heads(outs)
    assert np.all(got >= x.min(0) - 1e-12) and np.all(got <= x.max(0) + 1e-12)


def test_dominant_source_wins(oracle_mod):
    inp = make_merge_inputs("kimi", rows=2, seed=23, cp=4, H=4, D=16)
    lses = [np.zeros((2, 4)) for _ in range(4)]
    lses[2][:] = 200.0          # exp(-200) ~ 1e-87: the others vanish in fp64
    outs, lse_outs = oracle_mod.merge(inp.srcs, lses, True)
    assert np.array_equal(concat_heads(outs), widen_bf16(inp.srcs[2]))
    np.testing.assert_allclose(np.concatenate(lse_outs, 1), 200.0, rtol=1e-15)


# --- layout ---------------------------------------------------------------

def test_one_hot_head_routing(oracle_mod):
    # Head h goes to destination h // (H/cp) at local slot h % (H/cp)
    # ("[DCP] Run fi_a2a on FlashInfer's fused all-to-all + LSE reduce",
    # "Modifications"). Source j's payload encodes (j, b, h, d); for each
    # (b, h) exactly one source, k = (b + 3h) % cp, has a finite LSE, so the
    # merge must copy that source's encoded row to the routed position.
    cp, B, H, D = 4, 3, 8, 8
    Hl = H // cp
    srcs, lses = [], []
    for j in range(cp):
        s = np.empty((B, H, D))
        l = np.full((B, H), -np.inf)
        for b in range(B):
            for h in range(H):
                s[b, h] = [j * 1000 + b * 100 + h * 10 + d for d in range(D)]
                if (b + 3 * h) % cp == j:
                    l[b, h] = 0.25 * b - h
        srcs.append(s)
        lses.append(l)
    outs, lse_outs = oracle_mod.merge(srcs, lses, True, dtype="f64")
    for r in range(cp):
        for b in range(B):
            for i in range(Hl):
                h = r * Hl + i
                k = (b + 3 * h) % cp
                assert list(outs[r][b, i]) == [k * 1000 + b * 100 + h * 10 + d for d in range(D)]
                assert lse_outs[r][b, i] == 0.25 * b - h


def test_lse_strides_skip_padding(oracle_mod):
    # FlashMLA-style [B, H, 1] and padded LSE rows: the merge reads only
    # lse[b*row + h*head]; the padding holds NaN and must never be read.
    inp = make_merge_inputs("deepseek", rows=4, seed=29, cp=4, H=8, D=16)
    compact = [l.reshape(4, 8) for l in inp.lses]
    o0, l0 = oracle_mod.merge(inp.srcs, compact, True)
    padded = []
    for l in compact:
        p = np.full((4, 8, 3), np.nan, dtype=np.float32)  # row stride 24, head stride 3
        p[:, :, 0] = l
        padded.append(p.reshape(-1))
    o1, l1 = oracle_mod.merge(inp.srcs, padded, True, H=8, src_strides=(8 * 16, 16), lse_strides=(24, 3))
    for r in range(4):
        assert np.array_equal(o0[r], o1[r]) and np.array_equal(l0[r], l1[r])


def test_padded_source_rows(oracle_mod):
    # CUTLASS-style padded token stride ("[Attention] Add direct
    # symmetric-memory DCP A2A", commit notes): rows of H*D + pad elements,
    # the padding filled with NaN.
    inp = make_merge_inputs("kimi", rows=3, seed=31, cp=2, H=4, D=16)
    o0, l0 = oracle_mod.merge(inp.srcs, inp.lses, False)
    row = 4 * 16 + 48
    wide = []
    for s in inp.srcs:
        w = np.full((3, row), 0x7FC0, dtype=np.uint16)
        w[:, :64] = s.reshape(3, 64)
        wide.append(w.reshape(3, row // 16, 16))
    o1, l1 = oracle_mod.merge(wide, inp.lses, False, H=4, src_strides=(row, 16))
    for r in range(2):
        assert np.array_equal(o0[r], o1[r]) and np.array_equal(l0[r], l1[r])


def test_non_contiguous_head_storage(oracle_mod):
    # Heads taken from a wider backing array ("[Attention] Add direct
    # symmetric-memory DCP A2A", commit notes: non-contiguous 128-head backing
    # storage): head stride D + 24, row stride H * (D + 24); padding is NaN.
    inp = make_merge_inputs("kimi", rows=3, seed=37, cp=4, H=8, D=16)
    o0, l0 = oracle_mod.merge(inp.srcs, inp.lses, False)
    hs = 16 + 24
    wide = []
    for s in inp.srcs:
        w = np.full((3, 8, hs), 0x7FC0, dtype=np.uint16)
        w[:, :, :16] = s
        wide.append(w)
    o1, l1 = oracle_mod.merge(wide, inp.lses, False, H=8, D=16, src_strides=(8 * hs, hs))
    for r in range(4):
        assert np.array_equal(o0[r], o1[r]) and np.array_equal(l0[r], l1[r])


# --- the closed form: merged split attention = full attention ---------------

@pytest.mark.parametrize("split", ["halves", "interleaved", "four_uneven"])
@pytest.mark.parametrize("base_e", [True, False])
def test_merge_of_split_attention_is_full_attention(oracle_mod, split, base_e):
    from oracle.attention import attention, split_partials
    q, kv = tiny_qkv(seed=0)
    scale = 1.0 / math.sqrt(512)
    T = kv.shape[0]
    shards = {"halves": [np.arange(0, 32), np.arange(32, 64)],
              "interleaved": [np.arange(0, T, 2), np.arange(1, T, 2)],
              "four_uneven": [np.arange(0, 5), np.arange(5, 40), np.arange(40, 41), np.arange(41, 64)]}[split]
    o_parts, l_parts = split_partials(q, kv, shards, scale, base_e)
    o_full, l_full = attention(q, kv, scale, base_e)
    # 16 heads split over cp destinations
    outs, lse_outs = oracle_mod.merge(o_parts, l_parts, base_e, dtype="f64")
    np.testing.assert_allclose(concat_heads(outs), o_full, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(np.concatenate(lse_outs, 1), l_full, rtol=1e-13)


def test_empty_shard_in_split_attention(oracle_mod):
    # A shard that owns no tokens publishes lse = -inf ("[DCP] Optimize shared
    # Output, Query, and Indexer/Top-K via peer memory", commit notes) and must
    # leave the result equal to full attention.
    from oracle.attention import attention, split_partials
    q, kv = tiny_qkv(seed=0)
    scale = 1.0 / math.sqrt(512)
    shards = [np.arange(0, 64), np.arange(0, 0)]
    o_parts, l_parts = split_partials(q, kv, shards, scale)
    o_parts[1][:] = np.nan
    o_full, l_full = attention(q, kv, scale)
    outs, lse_outs = oracle_mod.merge(o_parts, l_parts, True, dtype="f64")
    np.testing.assert_allclose(concat_heads(outs), o_full, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(np.concatenate(lse_outs, 1), l_full, rtol=1e-15)


# --- seq_lens-driven empty-shard masking -----------------------------------------

def _masked_case(cp, interleave, lens, seed=0):
    """Partials of attention over each row's first lens[b] tokens, split over
    cp shards with the KV interleaved in blocks of `interleave` tokens. Empty
    shards get a NaN payload and a garbage (+7) LSE entry, which the mask must
    ignore. Returns (partials, lses, full attention o, full lse)."""
    from oracle.attention import attention
    q, kv = tiny_qkv(seed=seed)
    scale = 1.0 / math.sqrt(512)
    R, H, D = q.shape
    srcs = [np.empty((R, H, D)) for _ in range(cp)]
    lses = [np.empty((R, H)) for _ in range(cp)]
    o_full = np.empty((R, H, D))
    l_full = np.empty((R, H))
    for b in range(R):
        toks = np.arange(lens[b])
        for j in range(cp):
            own = toks[(toks // interleave) % cp == j]
            o, l = attention(q[b:b + 1], kv[own], scale)
            if own.size == 0:
                o[:] = np.nan
                l[:] = 7.0
            srcs[j][b], lses[j][b] = o[0], l[0]
        o, l = attention(q[b:b + 1], kv[toks], scale)
        o_full[b], l_full[b] = o[0], l[0]
    return srcs, lses, o_full, l_full


@pytest.mark.parametrize("cp,interleave,lens", [(4, 1, [1, 2, 64]), (4, 4, [3, 9, 17]), (2, 16, [5, 16, 40]),
                                                 (8, 2, [1, 15, 16])])
def test_seq_len_mask_gives_attention_over_the_row_context(oracle_mod, cp, interleave, lens):
    srcs, lses, o_full, l_full = _masked_case(cp, interleave, lens)
    outs, lse_outs = oracle_mod.merge(srcs, lses, True, dtype="f64", seq_lens=np.array(lens),
                                      interleave=interleave)
    np.testing.assert_allclose(concat_heads(outs), o_full, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(np.concatenate(lse_outs, 1), l_full, rtol=1e-13)


def test_zero_length_context_is_an_empty_row(oracle_mod):
    inp = make_merge_inputs("kimi", rows=3, seed=41, cp=4, H=8, D=16)
    outs, lse_outs = oracle_mod.merge(inp.srcs, inp.lses, False, seq_lens=np.array([0, 5, 0]), interleave=1)
    for r in range(4):
        assert np.array_equal(outs[r][[0, 2]], np.zeros((2, 2, 16)))
        assert np.all(lse_outs[r][[0, 2]] == -np.inf) and np.isfinite(lse_outs[r][1]).all()


def test_long_contexts_mask_nothing(oracle_mod):
    inp = make_merge_inputs("deepseek", rows=4, seed=43, cp=8, H=16, D=16)
    a, la = oracle_mod.merge(inp.srcs, inp.lses, True)
    b, lb = oracle_mod.merge(inp.srcs, inp.lses, True, seq_lens=np.array([64, 100, 1 << 20, 65]), interleave=8)
    for r in range(8):
        assert np.array_equal(a[r], b[r]) and np.array_equal(la[r], lb[r])


# --- the attention oracle (producer of the partials) ------------------------------

def test_attention_over_one_token_is_that_value():
    # softmax over a single token is 1: o = v, lse = s
    from oracle.attention import attention
    rng = np.random.default_rng(51)
    q = rng.standard_normal((2, 3, 576))
    kv = rng.standard_normal((1, 576))
    o, lse = attention(q, kv, 0.1, dv=512)
    assert np.array_equal(o, np.broadcast_to(kv[0, :512], (2, 3, 512)))
    np.testing.assert_allclose(lse, 0.1 * np.einsum("rhd,d->rh", q, kv[0]), rtol=1e-14)


def test_attention_with_zero_query_is_the_value_mean():
    # q = 0 gives equal scores: o = mean of the value rows, lse = log(T)
    from oracle.attention import attention
    rng = np.random.default_rng(53)
    kv = rng.standard_normal((37, 576))
    o, lse = attention(np.zeros((1, 2, 576)), kv, 0.3, dv=512)
    np.testing.assert_allclose(o[0, 1], kv[:, :512].mean(0), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, np.log(37.0), rtol=1e-15)
    _, lse2 = attention(np.zeros((1, 2, 576)), kv, 0.3, base_e=False, dv=512)
    np.testing.assert_allclose(lse2, np.log2(37.0), rtol=1e-15)


def test_attention_two_tokens_closed_form():
    # two tokens with scores 0 and ln 3: weights 1/4 and 3/4
    from oracle.attention import attention
    q = np.zeros((1, 1, 4)); q[0, 0, 0] = 1.0
    kv = np.array([[0.0, 1.0, 2.0, 9.0], [math.log(3.0), 5.0, -2.0, 9.0]])
    o, lse = attention(q, kv, 1.0, dv=3)
    np.testing.assert_allclose(o[0, 0], [0.75 * math.log(3.0), 0.25 * 1 + 0.75 * 5, 0.25 * 2 - 0.75 * 2], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(4.0), rtol=1e-15)


def test_attention_is_stable_for_widely_spread_scores():
    # scores 0 and 1000: exp(-1000) underflows to 0, so the second token takes
    # all the weight (o = its row exactly) and lse = 1000; taking the maximum
    # out before exponentiating is what keeps exp(1000) from overflowing
    from oracle.attention import attention
    q = np.zeros((1, 1, 4)); q[0, 0, 0] = 1.0
    kv = np.array([[0.0, 1.0, 2.0, 3.0], [1000.0, 5.0, -2.0, 7.0]])
    o, lse = attention(q, kv, 1.0, dv=4)
    assert np.array_equal(o[0, 0], kv[1])
    assert lse[0, 0] == 1000.0


def test_attention_is_invariant_under_token_permutation():
    from oracle.attention import attention
    rng = np.random.default_rng(55)
    q = rng.standard_normal((2, 4, 64)); kv = rng.standard_normal((20, 64))
    perm = rng.permutation(20)
    o1, l1 = attention(q, kv, 0.2, dv=48)
    o2, l2 = attention(q, kv[perm], 0.2, dv=48)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)
