"""Prefix lengths that live only in device memory (kvsel_desc.prefix_lens_dev).

A caller whose ragged lengths sit on the GPU (CompactAttention, 'Future directions':
page-table metadata built on the kernel side, with no CPU-GPU synchronisation) gives
the library a device array of lengths and a bound; every buffer is sized for the
bound, the data stays packed by the real lengths.  The whole path (scores, top-k,
compaction, block-union page table, cross-layer mean) must then give exactly what the
host-length calls give, and match the fp64 oracle.  A length beyond the bound, or one
the selection rules reject, is reported through the workspace error word and leaves
the outputs unwritten.
"""

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import kvsel as K
from attention_kv_cache_gb300 import synth as S
from oracle import kvsel_oracle as O
from tests.parity import assert_scores_close, assert_selection_equivalent, gathered_rows_match

pytestmark = pytest.mark.gpu


def _bound_buffers(inp, w, len_max, cuda):
    """q as usual; k, v packed by the real lengths inside buffers with room for every sequence at len_max."""
    from attention_kv_cache_gb300.pipeline import pack
    q, k, v = pack(inp, cuda)
    cap = w.batch * w.n_layers * w.h_kv * (len_max + w.window) * w.head_dim
    kb = torch.zeros(cap, dtype=torch.bfloat16, device=cuda)
    vb = torch.zeros(cap, dtype=torch.bfloat16, device=cuda)
    kb[:k.numel()] = k
    vb[:v.numel()] = v
    return q, kb, vb


def _run_both(w, len_max, cuda):
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    host = Pipeline(w, cuda)
    lens_dev = torch.tensor(w.prefix_lens, dtype=torch.int64, device=cuda)
    dev = Pipeline(w, cuda, lens_dev=lens_dev, len_max=len_max)
    qd, kd, vd = _bound_buffers(inp, w, len_max, cuda)
    mask = nkv = mask_d = nkv_d = None
    if w.block_union:
        mask = inp.mask.to(cuda)
        nkv = inp.n_kvblk
        pad = dev.n_kvblk_max - mask.shape[-1]
        mask_d = torch.nn.functional.pad(mask, (0, pad)).contiguous()
        nkv_d = torch.tensor(nkv, dtype=torch.int32, device=cuda)
    host.run(q, k, v, mask, nkv)
    dev.run(qd, kd, vd, mask_d, nkv_d)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(host.ws) == K.OK
    assert K.kvsel_read_device_error(dev.ws) == K.OK
    return inp, host, dev


def _assert_same(host, dev, w):
    n_tok = sum(w.n_layers * w.h_kv * L for L in w.prefix_lens)
    assert torch.equal(dev.scores[:n_tok], host.scores), "token scores differ from the host-length call's"
    if host.page_scores is not None:
        n_pg = host.page_scores.numel()
        assert torch.equal(dev.page_scores[:n_pg], host.page_scores), "page scores differ"
    if host.combined is not None:
        assert torch.equal(dev.combined[:host.combined.numel()], host.combined), "cross-layer scores differ"
    assert torch.equal(dev.idx, host.idx), "selections differ"
    assert torch.equal(dev.k_out, host.k_out) and torch.equal(dev.v_out, host.v_out), "compacted caches differ"
    if host.kv_indptr is not None:
        assert torch.equal(dev.kv_indptr, host.kv_indptr), "kv_indptr differs"
        n = int(host.kv_indptr[-1])
        assert torch.equal(dev.kv_indices[:n], host.kv_indices[:n]), "kv_indices differ"


def test_ragged_batch_lengths_on_device(cuda):
    """Ragged batch of three with the block-union table: lengths, and KV block counts, only on the device."""
    w = S.scaled(S.RAGGED_B8, n_layers=2, prefix_lens=[1500, 3333, 2048], k_keep=256)
    inp, host, dev = _run_both(w, 4100, cuda)
    _assert_same(host, dev, w)
    indptr_ref, indices_ref = O.block_union_csr(inp.mask.numpy(), w.h_kv, inp.n_kvblk)
    np.testing.assert_array_equal(dev.kv_indptr.cpu().numpy(), indptr_ref)
    np.testing.assert_array_equal(dev.kv_indices[:len(indices_ref)].cpu().numpy(), indices_ref)
    for b in range(w.batch):
        L = w.prefix_lens[b]
        ref = O.run_sequence(w, inp.q[b], inp.k[b], inp.v[b], with_gather=False)
        assert_scores_close(dev.token_scores(b), ref["pooled"], f"b{b} pooled scores")
        idx = dev.idx[b].cpu().numpy()
        for li in range(w.n_layers):
            for g in range(w.h_kv):
                assert_selection_equivalent(idx[li, g], ref["idx"][li, g], ref["pooled"][li, g], w.k_keep,
                                            f"b{b} l{li} g{g}")
                assert gathered_rows_match(dev.k_out[b, li, g], inp.k[b][li, g], idx[li, g], 1, L + w.window)


def test_paged_and_cross_layer_lengths_on_device(cuda):
    """Page mode (partial last page, recency pages) and the cross-layer mean with device lengths."""
    paged = S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200, 4099], k_keep=40)
    inp, host, dev = _run_both(paged, 9000, cuda)
    _assert_same(host, dev, paged)
    ref = O.run_sequence(paged, inp.q[1], inp.k[1], inp.v[1], with_gather=False)
    assert_scores_close(dev.page_view(1), ref["pages"], "paged b1 page scores")
    xl = S.scaled(S.LLAMA70B_64K_XLAYER, n_layers=4, prefix_lens=[2500, 1700], layer_range=(1, 3), k_keep=128)
    inp, host, dev = _run_both(xl, 2600, cuda)
    _assert_same(host, dev, xl)
    ref = O.run_sequence(xl, inp.q[1], inp.k[1], inp.v[1], with_gather=False)
    assert_scores_close(dev.combined_view(1), ref["pooled"], "cross-layer b1 combined")


def test_device_length_out_of_range_reported(cuda):
    """A device length above the bound, or a k the selection rules reject for one sequence: the call
    records KVSEL_ERR_INVALID_ARG in the error word and its kernels leave every output unwritten."""
    from attention_kv_cache_gb300.pipeline import Pipeline
    w = S.scaled(S.RAGGED_B8, n_layers=1, prefix_lens=[1000, 700], k_keep=64, block_union=False)
    inp = S.make_inputs(w, "cpu")
    q, k, v = _bound_buffers(inp, w, 1200, cuda)
    lens_dev = torch.tensor([1000, 1300], dtype=torch.int64, device=cuda)      # 1300 > bound 1200
    pipe = Pipeline(w, cuda, lens_dev=lens_dev, len_max=1200)
    pipe.scores.fill_(-7.0)
    pipe.idx.fill_(-3)
    pipe.k_out.fill_(5.0)
    pipe.run(q, k, v)
    assert K.kvsel_read_device_error(pipe.ws) == K.ERR_INVALID_ARG
    assert bool((pipe.scores == -7.0).all()) and bool((pipe.idx == -3).all()) and bool((pipe.k_out == 5.0).all())
    # lengths within the bound, but k = 64 > L for the second sequence: the selection is refused on the device
    lens_dev.copy_(torch.tensor([1000, 50], dtype=torch.int64))
    pipe.idx.fill_(-3)
    K.kvsel_select(pipe.desc, pipe.scores, w.n_layers * w.h_kv, 64, 0, True, pipe.idx, pipe.ws, pipe.ws_bytes)
    assert K.kvsel_read_device_error(pipe.ws) == K.ERR_INVALID_ARG
    assert bool((pipe.idx == -3).all())
    # and the same workspace serves a valid call afterwards
    lens_dev.copy_(torch.tensor([1000, 700], dtype=torch.int64))
    pipe.run(q, k, v)
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    assert bool((pipe.idx >= 0).all())


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_device_lengths_bit_equal(seed, cuda):
    """The random shapes of the fuzz tests with their lengths only on the device (bound a little above
    the longest): every output bit-equal to the host-length call's."""
    import random
    from tests.test_gpu_fuzz import draw
    w = draw(seed)
    len_max = max(w.prefix_lens) + random.Random(seed).choice([0, 1, 17, 300])
    inp, host, dev = _run_both(w, len_max, cuda)
    _assert_same(host, dev, w)
