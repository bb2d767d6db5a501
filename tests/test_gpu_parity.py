"""CUDA path against the fp64 oracle on the same seeded inputs (sizes the oracle finishes in seconds).

Every case spans several key tiles and segments and ends in a ragged tail.
"""

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import synth
from oracle import kvsel_oracle as O
from tests.parity import assert_scores_close, assert_selection_equivalent, gathered_rows_match

pytestmark = pytest.mark.gpu

S = synth
CASES = {
    # the tiny workload as specified
    "tiny": S.TINY,
    # LLaMA-shaped token mode, two layers, prefix not a multiple of any tile
    "llama_token": S.scaled(S.LLAMA8B_32K, n_layers=2, prefix_lens=[5003]),
    # paged: max over group, page max P = 16, last prefix page partial, recency 4
    "llama_paged": S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200]),
    # ragged batch of three with a block mask
    "ragged": S.scaled(S.RAGGED_B8, n_layers=2, prefix_lens=[1500, 3333, 2048], k_keep=256),
    # cross-layer L1 mean over layers 2..5 of 6, group of 8 (256 rows)
    "xlayer": S.scaled(S.LLAMA70B_64K_XLAYER, n_layers=6, prefix_lens=[3000], layer_range=(2, 5), k_keep=256),
    # edge shapes: d = 64, one window row, G = 1, no pooling
    "w1_g1_d64": S.Workload("edge_w1", 90, 2, 3, 3, 64, 1, (700,), group_reduce="sum", pool_k=1, k_keep=10),
    # full window of 64 rows, max reduce, widest pool
    "w64_pool63": S.Workload("edge_w64", 91, 1, 4, 2, 128, 64, (1777,), group_reduce="max", pool_k=63,
                             k_keep=100, n_clusters=4),
    # prefix of one token
    "L1": S.Workload("edge_L1", 92, 1, 4, 1, 128, 8, (1,), pool_k=7, k_keep=1),
    # max over heads whose window is not a power of two: each head padded to 32 tile rows (4 x 32 = 128)
    "w24_max_padded": S.Workload("edge_w24", 93, 2, 8, 2, 128, 24, (3000,), group_reduce="max", pool_k=5,
                                 k_keep=200, n_clusters=4),
    # W = 40 padded to 64 rows per head, group of 4: a 256-row tile with 24 dead rows in every head
    "w40_max_padded_rt256": S.Workload("edge_w40", 107, 1, 8, 2, 128, 40, (2345,), group_reduce="max", pool_k=7,
                                       k_keep=90, n_clusters=4),
    # W = 48 padded to 64 rows, group of 4 (256 tile rows), page mode with P = 16: the paired
    # epilogue over padded heads, page max of the pooled scores, recency pages
    "w48_max_padded_pages_rt256": S.Workload("edge_w48p", 112, 1, 8, 2, 128, 48, (4100,), group_reduce="max",
                                             pool_k=5, k_keep=24, page_size=16, n_recent=3, n_clusters=4),
    # W = 5 padded to 8 rows, group of 4, d = 64
    "w5_max_padded_d64": S.Workload("edge_w5", 108, 1, 8, 2, 64, 5, (3001,), group_reduce="max", pool_k=3,
                                    k_keep=40, n_clusters=4),
    # group of 10 with W = 24: 240 rows, but 10 x 32 padded rows exceed a 256-row tile, so the
    # CUDA-core kernels serve it
    "g10w24_max_cudacore": S.Workload("edge_g10w24", 109, 1, 20, 2, 128, 24, (1500,), group_reduce="max",
                                      pool_k=5, k_keep=100, n_clusters=4),
    # group of 6 x 32 rows = 192 rows in a 256-row tile: 64 padding rows must carry no mass
    "g6_rt256_padded": S.Workload("edge_g6", 98, 1, 12, 2, 128, 32, (2222,), group_reduce="sum", pool_k=7,
                                  k_keep=100, n_clusters=4),
    # group of 4 with the full 64-row window and max reduce: 256 rows, one head per 64 columns
    "g4w64_max_rt256": S.Workload("edge_g4w64", 105, 1, 8, 2, 128, 64, (1999,), group_reduce="max", pool_k=5,
                                  k_keep=80, n_clusters=4),
    # group of 32 heads with W = 8, max reduce, d = 64: 256 rows of 8-row heads
    "g32w8_max_d64_rt256": S.Workload("edge_g32w8", 106, 1, 32, 1, 64, 8, (700,), group_reduce="max", pool_k=3,
                                      k_keep=30),
    # group of 16 with W = 16 and max reduce (256 rows, head width below a warp)
    "g16w16_max": S.Workload("edge_g16", 94, 1, 16, 1, 64, 16, (2500,), group_reduce="max", pool_k=3,
                             k_keep=64, page_size=16, n_recent=2, n_clusters=4),
}


def run_case(w, cuda):
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    mask = nkv = None
    if w.block_union:
        mask = inp.mask.to(cuda)
        nkv = inp.n_kvblk
    pipe.run(q, k, v, mask, nkv)
    torch.cuda.synchronize()
    assert pipe.ws is not None
    from attention_kv_cache_gb300 import kvsel as K
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    return inp, pipe


@pytest.mark.parametrize("name", list(CASES))
def test_path_matches_oracle(name, cuda):
    w = CASES[name]
    inp, pipe = run_case(w, cuda)
    check_against_oracle(name, w, inp, pipe)


def check_against_oracle(name, w, inp, pipe):
    """Scores (pooled, raw, combined, pages), selections, compacted rows and the block-union table
    of one run of the pipeline against the oracle."""
    for b in range(w.batch):
        L = w.prefix_lens[b]
        ref = O.run_sequence(w, inp.q[b], inp.k[b], inp.v[b], with_gather=False)
        if w.layer_range is None:
            assert_scores_close(pipe.token_scores(b), ref["pooled"], f"{name} b{b} pooled scores")
        else:
            assert_scores_close(pipe.token_scores(b), ref["raw"], f"{name} b{b} raw scores")
            assert_scores_close(pipe.combined_view(b), ref["pooled"], f"{name} b{b} combined")
        if w.page_size > 1:
            assert_scores_close(pipe.page_view(b), ref["pages"], f"{name} b{b} page scores")
        idx = pipe.idx[b].cpu().numpy()
        for g in range(w.h_kv):
            for li in range(pipe.idx_layers):
                if w.layer_range is not None:
                    cand, rsel = ref["pooled"][g], ref["idx"][g]
                elif w.page_size > 1:
                    cand, rsel = ref["pages"][li, g][: -(-L // w.page_size) - w.n_recent], ref["idx"][li, g]
                else:
                    cand, rsel = ref["pooled"][li, g], ref["idx"][li, g]
                assert_selection_equivalent(idx[li, g], rsel, cand, w.k_keep, f"{name} b{b} l{li} g{g}")
        # the compacted cache holds exactly the selected rows (bytes), for every layer
        kb = inp.k[b]
        vb = inp.v[b]
        for layer in range(w.n_layers):
            for g in range(w.h_kv):
                sel = idx[0 if pipe.idx_layers == 1 else layer, g]
                assert gathered_rows_match(pipe.k_out[b, layer, g], kb[layer, g], sel, w.page_size, L + w.window)
                assert gathered_rows_match(pipe.v_out[b, layer, g], vb[layer, g], sel, w.page_size, L + w.window)
    if w.block_union:
        indptr, indices = O.block_union_csr(inp.mask.numpy(), w.h_kv, inp.n_kvblk)
        np.testing.assert_array_equal(pipe.kv_indptr.cpu().numpy(), indptr)
        got = pipe.kv_indices.cpu().numpy()[: indptr[-1]]
        np.testing.assert_array_equal(got, indices)


def test_long_context_two_pass_path(cuda):
    """640K-token prefix: each CTA's share no longer fits the single-read kernel's score buffer,
    so the two-pass tensor-core kernels run; checked against the oracle on the one unit."""
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = S.Workload("long_640k", 96, 1, 4, 1, 128, 32, (655360,), group_reduce="max", pool_k=7, page_size=16,
                   k_keep=128, n_recent=4, n_clusters=16)
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v)
    torch.cuda.synchronize()
    ref = O.run_sequence(w, inp.q[0], inp.k[0], with_gather=False)
    assert_scores_close(pipe.token_scores(0), ref["pooled"], "long pooled")
    assert_scores_close(pipe.page_view(0), ref["pages"], "long pages")
    n_cand = -(-w.prefix_lens[0] // 16) - w.n_recent
    assert_selection_equivalent(pipe.idx[0, 0, 0].cpu().numpy(), ref["idx"][0, 0], ref["pages"][0, 0][:n_cand],
                                w.k_keep, "long selection")


def test_unpooled_raw_scores(cuda):
    """pool_k = 1 gives the raw group column mass; sum mode mass of a group is at most G * W."""
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = S.scaled(S.LLAMA8B_32K, n_layers=1, prefix_lens=[3001], pool_k=1)
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.score(q, k)
    torch.cuda.synchronize()
    ref = O.run_sequence(w, inp.q[0], inp.k[0], with_gather=False)
    assert_scores_close(pipe.token_scores(0), ref["raw"], "raw")
    tot = pipe.token_scores(0).double().sum(-1).cpu()
    assert torch.all(tot <= w.group * w.window + 1e-3)
    assert K.kvsel_read_device_error(pipe.ws) == K.OK


def test_repeat_runs_bit_identical(cuda):
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = CASES["llama_paged"]
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v)
    a = (pipe.scores.clone(), pipe.page_scores.clone(), pipe.idx.clone(), pipe.k_out.clone())
    pipe.run(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a[0], pipe.scores) and torch.equal(a[1], pipe.page_scores)
    assert torch.equal(a[2], pipe.idx) and torch.equal(a[3], pipe.k_out)
