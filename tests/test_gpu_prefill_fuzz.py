"""Seeded random shapes for the causal prefill attention kernel against the fp64 oracle.

Each case draws the group shape (G = 1-8 query heads per KV head), the observation window, a batch
of one to three ragged prompts (lengths from a few rows to a dozen 128-row tiles, so that the last
tile is ragged and the tile pairs are uneven) and one or two layers; o, every row's lse, the
window rows' lse and the copied window queries are checked as in tests/test_gpu_prefill.py.
"""

import random

import pytest

from attention_kv_cache_gb300 import synth as S
from tests.test_gpu_prefill import _check_prefill, _run_prefill

pytestmark = pytest.mark.gpu

N_CASES = 12


def draw(seed: int) -> S.Workload:
    r = random.Random(7000 + seed)
    h_kv = r.choice([1, 2])
    G = r.choice([1, 2, 4, 8])
    W = r.choice([1, 4, 8, 16, 32])
    lens = tuple(r.randint(1, 1500) for _ in range(r.choice([1, 1, 2, 3])))
    return S.Workload(f"pf_fuzz{seed}", 400 + seed, r.choice([1, 2]), G * h_kv, h_kv, 128, W, lens, k_keep=1)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_prefill_matches_oracle(seed, cuda):
    w = draw(seed)
    inp, qf, k, v, o, lse, lse_win, q_win, desc, ws = _run_prefill(w, cuda)
    _check_prefill(w, inp, qf, o, lse, lse_win, q_win)
