"""Scoring variants and the CLAA schedule against the fp64 oracle (CUDA path through the C ABI).

Average pooling, the 'mean' group reduce, pre-softmax (logit) scores, all-head
selection shared by the KV heads, selections without the window, and the CLAA
prune schedule (per-layer selections plus the token-wise max over a layer
buffer), at sizes the oracle finishes in seconds that span several tiles and
segments with a ragged tail, and the variant workloads at full size.
"""

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import synth as S
from oracle import kvsel_oracle as O
from tests.parity import (WORST_LOGIT_RATIO, assert_scores_close, assert_selection_equivalent, gathered_rows_match,
                          logit_error_scale, pooled_bound)

pytestmark = pytest.mark.gpu

V = {
    # FastKV-style all-head selection with CLAA's average pooling, window of 8
    "allheads_avg_w8": S.scaled(S.LLAMA8B_32K, n_layers=2, prefix_lens=[5003], window=8, pool_type="avg",
                                head_reduce="all", k_keep=300),
    # GemFilter: last token's logits summed over all heads
    "gemfilter_w1": S.scaled(S.GEMFILTER_LLAMA8B_32K, n_layers=2, prefix_lens=[4099], k_keep=200),
    # LookaheadKV: mean over 32 rows per KV head, average pool, lookahead rows not kept
    "lookahead_mean": S.scaled(S.LOOKAHEAD_LLAMA8B_32K, n_layers=2, prefix_lens=[3001], k_keep=128),
    # logits per KV head, max pool, group sum
    "logits_group_w4": S.Workload("v_logits", 97, 2, 8, 2, 128, 4, (2777,), group_reduce="sum", pool_k=5,
                                  score_mode="logits", k_keep=50),
    # logits with the group max (signed maxima through order-preserving keys), d = 64
    "logits_groupmax_d64": S.Workload("v_logits_max", 98, 1, 8, 2, 64, 8, (1500,), group_reduce="max", pool_k=3,
                                      score_mode="logits", k_keep=40),
    # average pool in page mode: page max and page sum of the averaged scores
    "avg_pages_max": S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200], pool_type="avg"),
    "avg_pages_sum": S.scaled(S.LLAMA8B_128K_PAGED, n_layers=1, prefix_lens=[4100], pool_type="avg",
                              page_reduce="sum", k_keep=40),
    # average pool, group max with a window that is not a power of two (heads padded to 32 rows)
    "avg_padded_w24": S.Workload("v_avg_w24", 99, 1, 8, 2, 128, 24, (2000,), group_reduce="max", pool_k=7,
                                 pool_type="avg", k_keep=100, n_clusters=4),
    # logits, group max, W = 12 padded to 16 rows, group of 8
    "logits_groupmax_padded_w12": S.Workload("v_logits_max12", 110, 1, 16, 2, 128, 12, (2600,),
                                             group_reduce="max", pool_k=5, score_mode="logits", k_keep=60),
    # logits, group max, W = 40 padded to 64 rows, group of 3: 192 of 256 tile rows, so the paired
    # epilogue's last 64 columns are a head that exists only as padding and must be left out of the
    # signed maxima
    "logits_groupmax_padded_rt256": S.Workload("v_logits_max40", 113, 1, 6, 2, 128, 40, (2300,),
                                               group_reduce="max", pool_k=3, score_mode="logits", k_keep=48),
    # the CUDA-core kernels: group of 10 x 24 rows (padded beyond a 256-row tile), logits and average pool
    "logits_avg_cudacore_g10w24": S.Workload("v_cc_g10", 111, 1, 20, 2, 128, 24, (1300,), group_reduce="max",
                                             pool_k=7, pool_type="avg", score_mode="logits", k_keep=64),
    # logits summed over a group of 6 x 32 rows: 192 weighted rows and 64 padding rows in a 256-row tile
    "logits_rt256_padded": S.Workload("v_logits_256", 104, 1, 12, 2, 128, 32, (1900,), group_reduce="sum",
                                      pool_k=7, score_mode="logits", k_keep=64),
    # mean reduce over 256 padded rows (group of 8 x 32 rows), average pool
    "mean_rt256": S.Workload("v_mean_256", 100, 1, 16, 2, 128, 32, (2100,), group_reduce="mean", pool_k=7,
                             pool_type="avg", k_keep=64),
}


def _run(w, cuda):
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    return inp, pipe


@pytest.mark.parametrize("name", list(V))
def test_variant_matches_oracle(name, cuda):
    w = V[name]
    inp, pipe = _run(w, cuda)
    L, W = w.prefix_lens[0], w.window
    ref = O.run_sequence(w, inp.q[0], inp.k[0], inp.v[0], with_gather=False)
    idx = pipe.idx[0].cpu().numpy()
    braw = bpool = None
    if w.score_mode == "logits":
        braw = np.stack([logit_error_scale(inp.q[0][l], inp.k[0][l], w.group, L) for l in range(w.n_layers)])
        bpool = pooled_bound(braw.sum(axis=1) if w.head_reduce == "all" else braw, w.pool_k)
    if w.head_reduce == "all":
        assert_scores_close(pipe.token_scores(0), ref["raw"], f"{name} raw", bound=braw)
        agg = pipe.agg.view(w.n_layers, L)
        assert_scores_close(agg, ref["pooled"], f"{name} all-head pooled", bound=bpool)
        for li in range(w.n_layers):
            assert_selection_equivalent(idx[li, 0], ref["idx"][li], ref["pooled"][li], w.k_keep, f"{name} l{li}")
    else:
        assert_scores_close(pipe.token_scores(0), ref["pooled"], f"{name} pooled", bound=bpool)
        if w.page_size > 1:
            assert_scores_close(pipe.page_view(0), ref["pages"], f"{name} pages")
        for li in range(w.n_layers):
            for g in range(w.h_kv):
                if w.page_size > 1:
                    cand = ref["pages"][li, g][: -(-L // w.page_size) - w.n_recent]
                else:
                    cand = ref["pooled"][li, g]
                assert_selection_equivalent(idx[li, g], ref["idx"][li, g], cand, w.k_keep, f"{name} l{li} g{g}")
    assert idx.shape[-1] == w.n_sel()
    for li in range(w.n_layers):
        for g in range(w.h_kv):
            sel = idx[li, 0 if w.head_reduce == "all" else g]
            assert gathered_rows_match(pipe.k_out[0, li, g], inp.k[0][li, g], sel, w.page_size, L + W)
            assert gathered_rows_match(pipe.v_out[0, li, g], inp.v[0][li, g], sel, w.page_size, L + W)


def _claa_check(w, cuda, sample_layers=None):
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import ClaaPipeline, pack
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = ClaaPipeline(w, cuda)
    pipe.run(q, k, v)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    m, lp, nbuf, rate = w.claa
    L, W, G = w.prefix_lens[0], w.window, w.group
    ref = O.claa_sequence(inp.q[0], inp.k[0], L, W, G, w.h_kv, m, lp, nbuf, rate, w.pool_k, w.pool_type)
    assert pipe.k == ref["k"]
    lo, hi = ref["buffer"]
    assert pipe.buf_lo == lo - m
    for l in range(m, lp + 1):
        i = l - m
        raw = pipe.scores[i].double().sum(0).cpu().numpy()
        assert_scores_close(raw, ref["layer_scores"][l], f"claa layer {l} all-head score")
        u = O.pool(ref["layer_scores"][l], w.pool_k, w.pool_type)
        assert_scores_close(pipe.layer_scores[i], u, f"claa layer {l} pooled")
        assert_selection_equivalent(pipe.idx[0, i, 0].cpu().numpy(), ref["layer_idx"][l], u, ref["k"],
                                    f"claa layer {l} selection")
    assert_scores_close(pipe.prune_scores[0], ref["prune_scores"], "claa prune scores")
    assert_selection_equivalent(pipe.prune_idx[0, 0].cpu().numpy(), ref["prune_idx"], ref["prune_scores"], ref["k"],
                                "claa prune index")
    for l in (sample_layers or range(m, lp + 1)):
        sel = pipe.idx[0, l - m, 0].cpu().numpy()
        for g in range(w.h_kv):
            assert gathered_rows_match(pipe.k_out[0, l - m, g], inp.k[0][l, g], sel, 1, L + W)
            assert gathered_rows_match(pipe.v_out[0, l - m, g], inp.v[0][l, g], sel, 1, L + W)


def test_claa_schedule_small(cuda):
    w = S.scaled(S.CLAA_LLAMA8B_32K, n_layers=8, prefix_lens=[3000], claa=(2, 6, 3, 0.1))
    _claa_check(w, cuda)


def test_claa_schedule_buffer_clipped_at_defer(cuda):
    w = S.scaled(S.CLAA_LLAMA8B_32K, n_layers=5, prefix_lens=[1999], claa=(3, 4, 4, 0.25), pool_k=5)
    _claa_check(w, cuda)


def test_claa_full_size(cuda):
    """The 32K CLAA workload as specified: layers 4..15 scored, buffer 12..15, keep rate 0.2."""
    _claa_check(S.CLAA_LLAMA8B_32K, cuda, sample_layers=(4, 9, 15))


def test_gemfilter_full_size_sampled(cuda):
    w = S.GEMFILTER_LLAMA8B_32K
    inp, pipe = _run(w, cuda)
    L = w.prefix_lens[0]
    for layer in (0, 13, 31):
        raw = np.stack([O.score_unit(inp.q[0][layer], inp.k[0][layer], g, w.group, L, "sum", softmax=False)
                        for g in range(w.h_kv)])
        u = O.pool(O.head_sum(raw), w.pool_k, w.pool_type)
        b = pooled_bound(logit_error_scale(inp.q[0][layer], inp.k[0][layer], w.group, L).sum(axis=0), w.pool_k)
        assert_scores_close(pipe.agg.view(w.n_layers, L)[layer], u, f"gemfilter l{layer}", bound=b)
        want = O.select_tokens(u, w.k_keep, L, w.window)
        assert_selection_equivalent(pipe.idx[0, layer, 0].cpu().numpy(), want, u, w.k_keep, f"gemfilter sel {layer}")


def test_lookahead_full_size_sampled(cuda):
    w = S.LOOKAHEAD_LLAMA8B_32K
    inp, pipe = _run(w, cuda)
    L = w.prefix_lens[0]
    for layer, g in ((0, 0), (20, 3), (31, 7)):
        raw = O.score_unit(inp.q[0][layer], inp.k[0][layer], g, w.group, L, "mean")
        u = O.pool(raw, w.pool_k, w.pool_type)
        assert_scores_close(pipe.token_scores(0)[layer, g], u, f"lookahead l{layer} g{g}")
        want = O.select_tokens(u, w.k_keep, L, 0)
        assert_selection_equivalent(pipe.idx[0, layer, g].cpu().numpy(), want, u, w.k_keep, f"lookahead {layer} {g}")
        assert gathered_rows_match(pipe.k_out[0, layer, g], inp.k[0][layer, g], want, 1, L + w.window)


def test_zz_report_logit_error_ratio():
    """Reports the largest |gpu - oracle| / B over the pre-softmax cases above (B = logit_error_scale)."""
    print(f"\nworst pre-softmax error / B = {WORST_LOGIT_RATIO['ratio']:.3f} ({WORST_LOGIT_RATIO['what']})")
