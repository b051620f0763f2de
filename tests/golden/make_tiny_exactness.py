"""Writes tiny_exactness.json: the expected values of the tiny exactness check,
computed by the CPU oracle only (brute-force fp64 attention over the whole
64-token context).

Workload: cp = 2, 3 query rows, 16 heads, latent width 512; Q and the shared
latent K = V are N(0, 1) float32 from seed 0; scale 1/sqrt(512); no mask.
Run from the repository root:  python tests/golden/make_tiny_exactness.py
"""
import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from decode_context_mla_dcp_gb300.inputs import tiny_qkv  # noqa: E402  (seeded inputs only)
from oracle.attention import attention  # noqa: E402

SAMPLES = [(r, h, d) for r in range(3) for h in (0, 5, 8, 15) for d in (0, 1, 255, 511)]


def main():
    q, kv = tiny_qkv(seed=0)
    o, lse = attention(q, kv, 1.0 / math.sqrt(512), base_e=True)
    doc = {
        "what": "full-context fp64 attention for the tiny exactness check",
        "source": ("merge of split-softmax partials equals attention over the whole context: "
                   "'[DCP] Optimize shared Output, Query, and Indexer/Top-K via peer memory' "
                   "(sglang #32851), commit notes on permutation invariance and the cross-rank combine"),
        "written_by": "tests/golden/make_tiny_exactness.py (calls oracle.attention only)",
        "seed": 0, "rows": 3, "heads": 16, "d": 512, "tokens": 64, "scale": "1/sqrt(512)",
        "lse_base": "e",
        "lse": [[float(v) for v in row] for row in lse],
        "out_samples": [[r, h, d, float(o[r, h, d])] for (r, h, d) in SAMPLES],
        "out_row_sums": [[float(v) for v in row] for row in o.sum(axis=-1)],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_exactness.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
