"""Brute-force fp64 softmax attention over a latent KV: TEST INFRASTRUCTURE ONLY.

Used by the tests to build the split-context partials of the tiny exactness
check and to pin the merge against attention over the whole context.

What it follows:
* "[DCP] Optimize shared Output, Query, and Indexer/Top-K via peer memory"
  (sglang #32851), commit notes: under DCP the latent KV cache is interleaved
  across the ranks, each rank attends over the tokens it owns and returns a
  partial output plus its LSE, and attention is invariant to permuting the
  selected tokens; so any split of the tokens into shards, merged by LSE
  weight, gives attention over the whole set.
* "[DCP] Run fi_a2a on FlashInfer's fused all-to-all + LSE reduce"
  (sglang #40539), "Speed Tests and Profiling": MLA decode with a latent
  (kv_lora_rank) width of 512 shared by keys and values.

Decode rows see the whole context, so no causal mask is applied.
"""
from __future__ import annotations

import numpy as np

__all__ = ["attention", "split_partials"]


def attention(q: np.ndarray, kv: np.ndarray, scale: float, base_e: bool = True, dv: int | None = None):
    """Softmax attention of every query head over every token of ``kv``.

    q: [R, H, Dk] queries; kv: [T, Dk] latent rows. The key of token t is the
    whole row kv[t] (MLA: the 512-wide latent plus the 64-wide RoPE part); its
    value is the first ``dv`` entries (default: the whole row). Returns
    (o [R, H, dv], lse [R, H]) in float64, where s[r,h,t] = scale *
    <q[r,h], kv[t]>, o = sum_t softmax_t(s) kv[t, :dv] and
    lse = log(sum_t exp(s)) (log base 2 when base_e is False). An empty token
    set gives o = 0 and lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    R, H, _ = q.shape
    dv = kv.shape[1] if dv is None else dv
    if kv.shape[0] == 0:
        return np.zeros((R, H, dv)), np.full((R, H), -np.inf)
    s = scale * np.einsum("rhd,td->rht", q, kv)
    m = s.max(axis=-1, keepdims=True)   # log-sum-exp with the max taken out
    p = np.exp(s - m)
    z = p.sum(axis=-1)
    o = np.einsum("rht,td->rhd", p / z[..., None], kv[:, :dv])
    lse = m[..., 0] + np.log(z)
    if not base_e:
        lse = lse / np.log(2.0)
    return o, lse


def split_partials(q: np.ndarray, kv: np.ndarray, shards, scale: float, base_e: bool = True,
                   dv: int | None = None):
    """Per-shard attention: for each index array in ``shards``, attention over
    those tokens only. Returns lists (o_j [R, H, dv], lse_j [R, H])."""
    outs, lses = [], []
    for idx in shards:
        o, lse = attention(q, kv[np.asarray(idx, dtype=np.int64)], scale, base_e, dv)
        outs.append(o)
        lses.append(lse)
    return outs, lses
