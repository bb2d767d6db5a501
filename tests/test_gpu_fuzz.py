"""Seeded random shapes through the whole path, each against the oracle.

Each case draws a workload within the library's limits (d in {64, 128}, G W <= 256, W <= 64, page
mode with W a multiple of the page) from a seed: batch of one to three ragged prompts, group sizes
that pad their heads or their tile, every group reduce, pooling type and width, softmax or
pre-softmax scores, token or page mode, and cross-layer means.  The checks are those of the parity
tests (tests/test_gpu_parity.py): scores within the stated tolerance, selections equal up to the
near-tie rule, compacted rows and tables bit-exact.
"""

import random

import pytest

from attention_kv_cache_gb300 import synth as S
from tests.test_gpu_parity import check_against_oracle, run_case

pytestmark = pytest.mark.gpu

N_CASES = 48


def draw(seed: int) -> S.Workload:
    r = random.Random(1000 + seed)
    d = r.choice([64, 128])
    h_kv = r.choice([1, 2])
    page = r.random() < 0.3
    while True:
        G = r.choice([1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 32])
        W = r.choice([16, 32, 48, 64]) if page else r.choice([1, 2, 3, 5, 7, 8, 9, 12, 16, 17, 24, 31, 32, 40, 48, 63, 64])
        if G * W <= 256:
            break
    batch = r.choice([1, 1, 2, 3])
    lens = tuple(r.randint(1 if not page else 17, 3000) for _ in range(batch))
    n_layers = r.choice([1, 2, 3])
    xl = n_layers >= 2 and not page and r.random() < 0.3
    P = 16 if page else 1
    n_recent = 0
    if page:
        n_recent = r.choice([1, 2, 3])
        n_pages_min = min(-(-L // P) for L in lens)
        n_recent = min(n_recent, n_pages_min - 1)
        if n_recent < 1:                                   # too short for page mode: token mode
            page, P, n_recent = False, 1, 0
    if page:
        k_keep = r.randint(1, max(1, n_pages_min - n_recent))
    else:
        k_keep = r.randint(1, min(lens))
    score_mode = "logits" if r.random() < 0.25 else "softmax"
    return S.Workload(
        f"fuzz{seed}", 200 + seed, n_layers, G * h_kv, h_kv, d, W, lens,
        group_reduce=r.choice(["sum", "max", "mean"]), pool_k=r.choice([1, 3, 5, 7]), page_size=P,
        page_reduce=r.choice(["max", "sum"]) if page else "max", k_keep=k_keep, n_recent=n_recent,
        n_clusters=min(4, min(lens) // 256), layer_range=(0, n_layers - 1) if xl else None,
        pool_type=r.choice(["max", "avg"]), score_mode=score_mode)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape_matches_oracle(seed, cuda):
    w = draw(seed)
    inp, pipe = run_case(w, cuda)
    check_against_oracle(w.name, w, inp, pipe)
