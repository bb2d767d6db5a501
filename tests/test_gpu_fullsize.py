"""Full-size workloads in the configuration bench.py times, checked against the oracle on sampled units.

The whole path runs on the GPU over every layer and KV head; the oracle recomputes a few
(layer, KV head) units one by one from the same generated inputs (copied from the device), and
the compacted rows are compared byte for byte with the input rows the selection names.
"""

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import synth as S
from oracle import kvsel_oracle as O
from tests.parity import assert_scores_close, assert_selection_equivalent, gathered_rows_match

pytestmark = pytest.mark.gpu


def _run(w, cuda):
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    inp = S.make_inputs(w, str(cuda))
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    mask = inp.mask
    pipe.run(q, k, v, mask, inp.n_kvblk)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    return inp, pipe


def _check_unit(w, inp, pipe, b, layer, g, name):
    L, G, W = w.prefix_lens[b], w.group, w.window
    q_layer = inp.q[b][layer].cpu()
    k_unit = inp.k[b][layer, g].cpu()
    raw = O.score_unit(q_layer, _kv_view(k_unit, g, w.h_kv), g, G, L, w.group_reduce)
    pooled = O.max_pool(raw, w.pool_k)
    assert_scores_close(pipe.token_scores(b)[layer, g], pooled, f"{name} pooled l{layer} g{g}")
    sel = pipe.idx[b, layer, g].cpu().numpy()
    if w.page_size == 1:
        want = O.select_tokens(pooled, w.k_keep, L, W)
        assert_selection_equivalent(sel, want, pooled, w.k_keep, f"{name} sel l{layer} g{g}")
    else:
        U = O.page_reduce(pooled, w.page_size, w.page_reduce)
        assert_scores_close(pipe.page_view(b)[layer, g], U, f"{name} pages l{layer} g{g}")
        want = O.select_pages(U, w.k_keep, w.n_recent, L, W, w.page_size)
        n_cand = -(-L // w.page_size) - w.n_recent
        assert_selection_equivalent(sel, want, U[:n_cand], w.k_keep, f"{name} sel l{layer} g{g}")
    assert gathered_rows_match(pipe.k_out[b, layer, g], inp.k[b][layer, g], sel, w.page_size, L + W)
    assert gathered_rows_match(pipe.v_out[b, layer, g], inp.v[b][layer, g], sel, w.page_size, L + W)


class _kv_view:
    """Stands in for a [h_kv, N, d] layer tensor whose only needed entry is head g."""

    def __init__(self, k_unit, g, h_kv):
        self.k, self.g = k_unit, g

    def __getitem__(self, i):
        assert i == self.g
        return self.k


@pytest.mark.parametrize("wname", ["llama8b_32l_h32x8_d128_L32768_W32",
                                   "llama8b_32l_h32x8_d128_L131072_W32_paged16"])
def test_full_size_sampled_units(wname, cuda):
    w = S.by_name(wname)
    inp, pipe = _run(w, cuda)
    for layer, g in ((0, 0), (17, 5), (31, 7)):
        _check_unit(w, inp, pipe, 0, layer, g, wname)


def test_full_size_ragged_batch(cuda):
    w = S.RAGGED_B8
    inp, pipe = _run(w, cuda)
    for b, layer, g in ((0, 0, 0), (3, 20, 6), (7, 31, 7)):
        _check_unit(w, inp, pipe, b, layer, g, "ragged")
    indptr, indices = O.block_union_csr(inp.mask.cpu().numpy(), w.h_kv, inp.n_kvblk)
    np.testing.assert_array_equal(pipe.kv_indptr.cpu().numpy(), indptr)
    np.testing.assert_array_equal(pipe.kv_indices.cpu().numpy()[: indptr[-1]], indices)


def test_full_size_cross_layer_one_head(cuda):
    """70B-shaped: the combined score of one KV head needs its 72 layers; the oracle recomputes them all."""
    w = S.LLAMA70B_64K_XLAYER
    inp, pipe = _run(w, cuda)
    g = 3
    L, G = w.prefix_lens[0], w.group
    lo, hi = w.layer_range
    raw = np.stack([O.score_unit(inp.q[0][layer].cpu(), _kv_view(inp.k[0][layer, g].cpu(), g, w.h_kv), g, G, L,
                                 w.group_reduce) for layer in range(lo, hi + 1)])
    for i, layer in enumerate((lo, (lo + hi) // 2, hi)):
        assert_scores_close(pipe.token_scores(0)[layer, g], raw[layer - lo], f"xlayer raw l{layer}")
    S_ = O.cross_layer_mean(raw, 0, hi - lo)
    u = O.max_pool(S_, w.pool_k)
    assert_scores_close(pipe.combined_view(0)[g], u, "xlayer combined")
    sel = pipe.idx[0, 0, g].cpu().numpy()
    assert_selection_equivalent(sel, O.select_tokens(u, w.k_keep, L, w.window), u, w.k_keep, "xlayer sel")
    for layer in (0, 40, 79):
        assert gathered_rows_match(pipe.k_out[0, layer, g], inp.k[0][layer, g], sel, 1, L + w.window)
        assert gathered_rows_match(pipe.v_out[0, layer, g], inp.v[0][layer, g], sel, 1, L + w.window)
