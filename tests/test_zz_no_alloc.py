"""kvsel_score_noalloc: scoring for callers that cannot allocate device memory.

Some callers have no way to get a workspace: a plugin running inside a host
program that owns all of the GPU's memory, or a latency-critical caller that
must not pay cudaMalloc's device-wide synchronisation.  kvsel_score_noalloc
serves them with scratch that lives inside the library.  These tests call it
through the C ABI and check that it returns exactly what kvsel_score (the
entry point with a caller-provided workspace) returns — both run the same
deterministic kernels — on two calls in a row with different shapes, so that
whatever the first call leaves in the shared scratch cannot leak into the
second, and that the scratch's error word reads back clean after each.

This file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

from attention_kv_cache_gb300 import kvsel as K
from attention_kv_cache_gb300 import synth as S


def test_oversized_request_rejected_before_any_launch():
    # 200 layers x 8 KV heads at 128K needs far more than the built-in scratch
    d = K.make_desc(n_layers=200, h_q=32, h_kv=8, head_dim=128, window=32, prefix_lens=[131072])
    assert K.kvsel_workspace_size(d) > K.NOALLOC_SCRATCH_BYTES
    assert K.raw_call("kvsel_score_noalloc", ctypes.byref(d), 16, 16, 16, None, None) == K.ERR_WORKSPACE
    bad = K.make_desc(n_layers=1, h_q=4, h_kv=2, head_dim=96, window=16, prefix_lens=[512])
    assert K.raw_call("kvsel_score_noalloc", ctypes.byref(bad), 16, 16, 16, None, None) == K.ERR_UNSUPPORTED


def test_misaligned_pointer_rejected_before_anything_is_enqueued():
    # the argument checks run before the error word is cleared: nothing reaches a stream
    d = K.make_desc(n_layers=1, h_q=4, h_kv=2, head_dim=64, window=16, prefix_lens=[512])
    before = K.kvsel_launch_count()
    assert K.raw_call("kvsel_score_noalloc", ctypes.byref(d), 24, 16, 16, None, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_score_noalloc", ctypes.byref(d), 16, 16, None, None, None) == K.ERR_INVALID_ARG
    paged = K.make_desc(n_layers=1, h_q=4, h_kv=2, head_dim=64, window=16, prefix_lens=[512], page_size=16)
    assert K.raw_call("kvsel_score_noalloc", ctypes.byref(paged), 16, 16, 16, None, None) == K.ERR_INVALID_ARG
    assert K.kvsel_launch_count() == before


def _scores_both_ways(w, cuda):
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    inp = S.make_inputs(w, "cpu")
    q, k, _ = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.score(q, k)                                   # kvsel_score with a torch-allocated workspace
    ref_scores = pipe.scores.clone()
    ref_pages = pipe.page_scores.clone() if pipe.page_scores is not None else None
    out = torch.full_like(pipe.scores, float("nan"))
    pages = torch.full_like(pipe.page_scores, float("nan")) if pipe.page_scores is not None else None
    K.kvsel_score_noalloc(pipe.desc_score, q, k, out, pages)
    assert K.kvsel_noalloc_read_device_error() == K.OK
    torch.cuda.synchronize()
    return ref_scores, ref_pages, out, pages


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice(cuda):
    first = S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200])       # page mode, max reduce
    second = S.scaled(S.RAGGED_B8, n_layers=1, prefix_lens=[1500, 3333], block_union=False)  # ragged, sum
    for w in (first, second):
        ref_scores, ref_pages, out, pages = _scores_both_ways(w, cuda)
        assert torch.equal(out, ref_scores), f"{w.name}: token scores differ from kvsel_score's"
        if ref_pages is not None:
            assert torch.equal(pages, ref_pages), f"{w.name}: page scores differ from kvsel_score's"
