"""The seeded input generator: reproducible, and drawing the stated laws."""
import numpy as np
import pytest
import torch

from decode_context_mla_dcp_gb300.inputs import (BF16_QNAN, CONFIGS, bf16_bits, f16_bits,
                                                 make_merge_inputs, tiny_qkv)


def test_same_seed_same_bytes():
    a = make_merge_inputs("spec", rows=16, seed=4)
    b = make_merge_inputs("spec", rows=16, seed=4)
    c = make_merge_inputs("spec", rows=16, seed=5)
    for j in range(a.cp):
        assert np.array_equal(a.srcs[j], b.srcs[j]) and np.array_equal(a.lses[j], b.lses[j], equal_nan=True)
    assert not np.array_equal(a.srcs[0], c.srcs[0])


def test_sources_draw_independent_streams():
    a = make_merge_inputs("kimi", rows=4, seed=0)
    assert not np.array_equal(a.srcs[0], a.srcs[1])


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        # exact ties between two bf16 values, both parities
                        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
                        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_bits(x), ref)
    assert bf16_bits(np.array([np.nan], dtype=np.float32))[0] == BF16_QNAN


def test_f16_rounding_matches_torch():
    x = np.random.default_rng(1).standard_normal(10000).astype(np.float32) * 100
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f16_bits(x), ref)


def test_kimi_law_and_layout():
    inp = make_merge_inputs("kimi", rows=128, seed=0)
    assert inp.cp == 4 and inp.H == 64 and inp.D == 512 and not inp.lse_base_e
    l = np.stack(inp.lses)
    assert l.shape == (4, 128, 64) and l.min() >= -4 and l.max() <= 24
    assert abs(l.mean() - 10.0) < 0.2
    x = np.stack(inp.srcs)
    vals = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(vals.mean()) < 0.01 and abs(vals.std() - 1) < 0.01


def test_deepseek_flashmla_lse_layout_and_law():
    inp = make_merge_inputs("deepseek", rows=64, seed=0)
    assert inp.lses[0].shape == (64, 128, 1) and inp.lse_stride == 128 and inp.lse_base_e
    l = np.stack(inp.lses)
    assert abs(l.mean() - 12) < 0.1 and abs(l.std() - 4) < 0.1


def test_spec_decode_empty_shards():
    inp = make_merge_inputs("spec", rows=1024, seed=0)
    assert inp.empty.shape == (1024, 4)
    assert 0.08 < inp.empty.mean() < 0.12
    for j in range(4):
        e = inp.empty[:, j]
        assert np.all(inp.lses[j][e] == -np.inf)
        assert np.all(inp.srcs[j][e] == BF16_QNAN)
        assert np.isfinite(inp.lses[j][~e]).all()
    finite = np.concatenate([inp.lses[j][~inp.empty[:, j]].ravel() for j in range(4)])
    assert abs(finite.mean() - 10) < 0.1 and abs(finite.std() - 6) < 0.1


def test_stress_config_shape():
    cfg = CONFIGS["stress"]
    assert (cfg.cp, cfg.H, cfg.D, cfg.rows) == (8, 128, 512, (4096,))
    inp = make_merge_inputs("stress", rows=2, seed=0)
    l = np.stack(inp.lses)
    assert l.min() >= 0 and l.max() <= 30


def test_tiny_qkv_shapes():
    q, kv = tiny_qkv(0)
    assert q.shape == (3, 16, 512) and kv.shape == (64, 512) and q.dtype == np.float32


def test_golden_tiny_fixture_matches_oracle():
    import json
    import math
    import os
    from oracle.attention import attention
    doc = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_exactness.json")))
    q, kv = tiny_qkv(doc["seed"])
    o, lse = attention(q, kv, 1 / math.sqrt(512))
    np.testing.assert_allclose(lse, np.array(doc["lse"]), rtol=1e-14)
    for r, h, d, v in doc["out_samples"]:
        assert o[r, h, d] == pytest.approx(v, rel=1e-12, abs=1e-14)
    np.testing.assert_allclose(o.sum(-1), np.array(doc["out_row_sums"]), rtol=1e-12, atol=1e-12)
