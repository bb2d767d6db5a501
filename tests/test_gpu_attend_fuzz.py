"""Seeded random shapes for attention over a selection, read in place, against the fp64 oracle.

Each case draws the group shape (query rows per table row R = G n_q from 1 to 32: the warp
kernels up to 8, the block kernel above), d, the block size (multiples of 16 take the TMA kernel,
others the copy kernel), the prompt length and the table: a uniform list per row, a CSR table with
rows of different lengths (empty ones included), or every block of the cache.  Block ids may repeat
and come in any order; all lie in the cache.
"""

import random

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import synth as S
from tests.test_gpu_attend import _close, _ref, _ws

pytestmark = pytest.mark.gpu

N_CASES = 24


def draw(seed: int):
    r = random.Random(5000 + seed)
    while True:
        h_kv = r.choice([1, 2])
        G = r.choice([1, 2, 3, 4, 6, 8, 16])
        n_q = r.choice([1, 1, 2, 3, 4])
        if G * n_q <= 32:
            break
    d = r.choice([64, 128])
    P = r.choice([1, 4, 8, 16, 16, 32, 48, 64])
    L = r.randint(1, 2500)
    W = r.choice([1, 4, 8])
    mode = r.choice(["uniform", "csr", "whole"])
    return h_kv, G, n_q, d, P, L, W, mode, r


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_attention_matches_oracle(seed, cuda):
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import pack
    h_kv, G, n_q, d, P, L, W, mode, r = draw(seed)
    n_layers = 2
    w = S.Workload(f"attn_fuzz{seed}", 300 + seed, n_layers, G * h_kv, h_kv, d, W, (L,), k_keep=1)
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    desc = K.make_desc(n_layers=n_layers, h_q=G * h_kv, h_kv=h_kv, head_dim=d, window=W, prefix_lens=[L])
    n_blocks = -(-(L + W) // P)
    rows = n_layers * h_kv
    g = torch.Generator().manual_seed(seed)
    qd = S.make_decode_queries(w, n_q, "cpu")
    o = torch.full((1, n_layers, G * h_kv, n_q, d), float("nan"), dtype=torch.float32, device=cuda)
    if mode == "whole":
        lists = [[list(range(n_blocks)) for _ in range(h_kv)] for _ in range(n_layers)]
        ws = _ws(K, K.kvsel_attend_workspace_size(desc, n_q, P, n_blocks), cuda)
        K.kvsel_attend(desc, qd.to(cuda), n_q, k, v, None, None, 0, P, n_blocks, o, ws)
    elif mode == "uniform":
        n_per = r.randint(1, min(64, 2 * n_blocks))
        ids = torch.randint(0, n_blocks, (rows, n_per), generator=g, dtype=torch.int32)
        lists = ids.view(n_layers, h_kv, n_per).tolist()
        ws = _ws(K, K.kvsel_attend_workspace_size(desc, n_q, P, n_per), cuda)
        K.kvsel_attend(desc, qd.to(cuda), n_q, k, v, None, ids.to(cuda), n_per, P, n_per, o, ws)
    else:
        lens = [r.choice([0, r.randint(1, min(80, 2 * n_blocks))]) for _ in range(rows)]
        if sum(lens) == 0:
            lens[0] = 1
        indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        ids = torch.randint(0, n_blocks, (int(indptr[-1]),), generator=g, dtype=torch.int32)
        flat = ids.tolist()
        lists = [[flat[indptr[l * h_kv + gg]:indptr[l * h_kv + gg + 1]] for gg in range(h_kv)] for l in range(n_layers)]
        mb = max(lens)
        ws = _ws(K, K.kvsel_attend_workspace_size(desc, n_q, P, mb), cuda)
        K.kvsel_attend(desc, qd.to(cuda), n_q, k, v, torch.from_numpy(indptr).to(cuda), ids.to(cuda), 0, P, mb, o, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    _close(o[0], _ref(w, qd[0], inp.k[0], inp.v[0], lists, P, n_q),
           f"seed {seed}: R={G * n_q} d={d} P={P} L={L} {mode}")
