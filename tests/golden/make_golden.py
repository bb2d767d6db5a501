"""Writes tests/golden/formula_case.json from the fp64 oracle alone.

The inputs are closed-form (no random numbers), rounded to bf16, so any
machine can rebuild them:  q[h, j, c] = sin(1 + 0.7 h + 1.3 j + 0.37 c) * 2,
k[g, t, c] = cos(0.5 + 1.1 g + 0.29 t + 0.53 c) * 1.5.  The shapes are a
miniature of the LLaMA-shaped workloads: H_q = 4, H_kv = 2, d = 64, L = 40,
W = 4, group sum, max-pool 7, top-8 tokens + window.

Run:  python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
from oracle import kvsel_oracle as O  # noqa: E402

HQ, HKV, D, L, W, K = 4, 2, 64, 40, 4, 8


def formula_inputs():
    h = np.arange(HQ)[:, None, None]; j = np.arange(W)[None, :, None]; c = np.arange(D)[None, None, :]
    q = np.sin(1.0 + 0.7 * h + 1.3 * j + 0.37 * c) * 2.0
    g = np.arange(HKV)[:, None, None]; t = np.arange(L + W)[None, :, None]
    k = np.cos(0.5 + 1.1 * g + 0.29 * t + 0.53 * c) * 1.5
    q = torch.from_numpy(q).to(torch.bfloat16)
    k = torch.from_numpy(k).to(torch.bfloat16)
    return q, k


def expected():
    q, k = formula_inputs()
    G = HQ // HKV
    raw = np.stack([O.score_unit(q, k, g, G, L, "sum") for g in range(HKV)])
    pooled = O.max_pool(raw, 7)
    idx = np.stack([O.select_tokens(pooled[g], K, L, W) for g in range(HKV)])
    return raw, pooled, idx


if __name__ == "__main__":
    raw, pooled, idx = expected()
    out = {
        "about": "Formula inputs (see make_golden.py); expected values from the fp64 oracle. "
                 "Scoring follows ClusterAttn 'Background and key observations' (masked window softmax, "
                 "column sum over the window rows, prefix columns) with CLAA decision 2's sum over the "
                 "group's heads and 1-D pooling of width 7.",
        "shape": {"h_q": HQ, "h_kv": HKV, "d": D, "L": L, "W": W, "k": K, "pool_k": 7, "reduce": "sum"},
        "raw": [[float(x) for x in r] for r in raw],
        "pooled": [[float(x) for x in r] for r in pooled],
        "idx": [[int(x) for x in r] for r in idx],
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "formula_case.json"), "w") as f:
        json.dump(out, f, indent=1)
