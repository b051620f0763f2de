"""Seeded synthetic inputs for the DCP LSE-weighted merge.

This module only draws random numbers and lays them out; it holds none of the
merge's arithmetic. Both the CUDA path and the CPU oracle are fed from the same
host arrays it returns, so they see identical bytes.

Workload shapes follow the pages:
* Kimi-K2.5 geometry, "[Attention] Add direct symmetric-memory DCP A2A"
  (vLLM #48897), "A2A + LSE-reduce latency reduction": 64 heads in total,
  16 per rank (cp = 4), head dimension 512, bf16.
* DeepSeek-V2 geometry, "[DCP] Run fi_a2a on FlashInfer's fused all-to-all +
  LSE reduce" (sglang #40539), "Speed Tests and Profiling": TP 8 = DCP 8,
  16 heads per rank, head dimension 512, FlashMLA's [B, H, 1] LSE.
* Speculative decoding rows = requests x verify tokens (same page,
  "Modifications"); empty context shards publish LSE = -inf
  ("[Attention] Add direct symmetric-memory DCP A2A", commit notes).

Distributions (the pages give none; these are the synthetic stand-ins):
partials are bf16-rounded N(0, 1); LSEs are fp32 from the per-config law
below ("N(mu, s)" means mean mu, standard deviation s). Every tensor draws
from its own stream, keyed by (seed, kind, source index).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = ["MergeConfig", "MergeInputs", "CONFIGS", "bf16_bits", "f16_bits",
           "make_merge_inputs", "tiny_qkv", "rng_for", "make_mla_inputs", "MLA_SCALE"]

_KIND_PAYLOAD, _KIND_LSE, _KIND_EMPTY, _KIND_Q, _KIND_KV, _KIND_MLA_Q, _KIND_MLA_KV = 1, 2, 3, 4, 5, 6, 7

# DeepSeek-V2 MLA scores are scaled by 1/sqrt(qk_nope + qk_rope) = 1/sqrt(128 + 64)
# before absorption; the absorbed 576-wide keys keep that scale.
MLA_SCALE = 192 ** -0.5

BF16_QNAN = 0x7FC0
F16_QNAN = 0x7E00


@dataclass(frozen=True)
class MergeConfig:
    name: str
    cp: int
    H: int                  # total heads; each destination owns H // cp
    D: int
    rows: tuple             # batch rows swept
    lse_base_e: bool
    lse_law: tuple          # ("uniform", lo, hi) or ("normal", mean, std)
    lse_layout: str = "BH"  # "BH" = [B, H]; "BH1" = FlashMLA [B, H, 1]
    p_empty: float = 0.0    # probability that a (row, shard) is an empty shard


CONFIGS = {
    # cp=4, 64 heads, base-2 LSE U[-4, 24]
    "kimi": MergeConfig("kimi-k2.5", 4, 64, 512, (1, 8, 16, 32, 64, 128), False, ("uniform", -4.0, 24.0)),
    # cp=8, 128 heads, base-e LSE N(12, 4) in [B, H, 1]
    "deepseek": MergeConfig("deepseek-v2", 8, 128, 512, (1, 2, 4, 8, 16, 32, 64, 128), True,
                            ("normal", 12.0, 4.0), "BH1"),
    # 256 requests x 4 verify tokens, cp=4, 64 heads, base-e N(10, 6), 10% empty (row, shard)
    "spec": MergeConfig("spec-decode-256x4", 4, 64, 512, (1024,), True, ("normal", 10.0, 6.0), p_empty=0.1),
    # cp=8, 128 heads, 4096 rows, base-e U[0, 30]
    "stress": MergeConfig("bandwidth-stress", 8, 128, 512, (4096,), True, ("uniform", 0.0, 30.0)),
}


@dataclass
class MergeInputs:
    cp: int
    B: int
    H: int
    D: int
    lse_base_e: bool
    srcs: list              # cp x np.uint16 [B, H, D] (raw bf16 or f16 bits)
    lses: list              # cp x np.float32 [B, H] or [B, H, 1]
    lse_stride: int         # elements between rows of an LSE array
    dtype: str = "bf16"
    empty: np.ndarray | None = field(default=None)  # [B, cp] bool: empty (row, shard)


def rng_for(seed: int, kind: int, index: int = 0) -> np.random.Generator:
    """Independent stream per (seed, tensor kind, source index)."""
    return np.random.default_rng(np.random.SeedSequence([seed, kind, index]))


def bf16_bits(x: np.ndarray, chunk: int = 1 << 24) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns the
    16-bit patterns. NaN becomes the canonical quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for s in range(0, flat.size, chunk):
        u = flat[s:s + chunk].view(np.uint32)
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        r = r.astype(np.uint16)
        nan = np.isnan(flat[s:s + chunk])
        if nan.any():
            r[nan] = BF16_QNAN
        out[s:s + chunk] = r
    return out.reshape(x.shape)


def f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to IEEE binary16 (numpy's conversion, ties to even)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _draw_lse(rng: np.random.Generator, law: tuple, shape) -> np.ndarray:
    kind, a, b = law
    if kind == "uniform":
        return rng.uniform(a, b, size=shape).astype(np.float32)
    if kind == "normal":
        return (a + b * rng.standard_normal(size=shape)).astype(np.float32)
    raise ValueError(f"unknown LSE law {kind!r}")


def make_merge_inputs(cfg: MergeConfig | str, rows: int, seed: int = 0, dtype: str = "bf16",
                      p_empty: float | None = None, H: int | None = None, cp: int | None = None,
                      D: int | None = None) -> MergeInputs:
    """Draw one batch of cp partial outputs and LSEs for ``rows`` batch rows.

    For an empty (row, shard) every head's LSE is -inf and the payload is
    filled with NaN: a merge that reads or weights it leaks NaN.
    Overrides (H, cp, D, p_empty) serve the odd-shape tests.
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    cp = cfg.cp if cp is None else cp
    H = cfg.H if H is None else H
    D = cfg.D if D is None else D
    p_empty = cfg.p_empty if p_empty is None else p_empty
    B = int(rows)
    to_bits = bf16_bits if dtype == "bf16" else f16_bits
    qnan = BF16_QNAN if dtype == "bf16" else F16_QNAN

    empty = None
    if p_empty > 0:
        empty = rng_for(seed, _KIND_EMPTY).random(size=(B, cp)) < p_empty

    srcs, lses = [], []
    for j in range(cp):
        payload = to_bits(rng_for(seed, _KIND_PAYLOAD, j).standard_normal(size=(B, H, D), dtype=np.float32))
        lse = _draw_lse(rng_for(seed, _KIND_LSE, j), cfg.lse_law, (B, H))
        if empty is not None:
            rows_j = empty[:, j]
            payload[rows_j] = qnan
            lse[rows_j] = -np.inf
        if cfg.lse_layout == "BH1":
            lse = lse.reshape(B, H, 1)
        srcs.append(payload)
        lses.append(lse)
    return MergeInputs(cp=cp, B=B, H=H, D=D, lse_base_e=cfg.lse_base_e, srcs=srcs, lses=lses,
                       lse_stride=H, dtype=dtype, empty=empty)


def tiny_qkv(seed: int = 0, rows: int = 3, heads: int = 16, d: int = 512, tokens: int = 64):
    """Tiny exactness check: queries [rows, heads, d] and a latent K = V of
    [tokens, d], both N(0, 1) float32."""
    q = rng_for(seed, _KIND_Q).standard_normal(size=(rows, heads, d), dtype=np.float32)
    kv = rng_for(seed, _KIND_KV).standard_normal(size=(tokens, d), dtype=np.float32)
    return q, kv


def make_mla_inputs(B: int, H: int, T: int, Dk: int = 576, seed: int = 0):
    """Decode queries and one shard's latent KV cache, bf16 bit patterns of
    N(0, 1) draws: q [B, H, Dk] and kv [B, T, Dk] (row b's shard-local
    tokens)."""
    q = bf16_bits(rng_for(seed, _KIND_MLA_Q).standard_normal(size=(B, H, Dk), dtype=np.float32))
    kv = bf16_bits(rng_for(seed, _KIND_MLA_KV).standard_normal(size=(B, T, Dk), dtype=np.float32))
    return q, kv
