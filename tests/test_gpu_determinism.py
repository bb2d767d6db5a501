"""Bit-determinism: the same inputs give the same bits, call after call.

Every output of the path (token and page scores, cross-layer scores, selections, compacted rows,
block-union tables, attention over the selection) is compared bit for bit between two runs of the
same pipeline.  The kernels make this hold by construction: partial sums meet in a fixed order
(or, where shared-memory atomics join them, as exactly two addends, whose sum does not depend on
their order), maxima are exact, and the work split depends only on the shapes.
"""

import pytest
import torch

from attention_kv_cache_gb300 import kvsel as K
from attention_kv_cache_gb300 import synth as S

pytestmark = pytest.mark.gpu

CASES = {
    "paged_max": S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200]),
    "token_sum": S.scaled(S.LLAMA8B_32K, n_layers=2, prefix_lens=[5003]),
    "ragged_csr": S.scaled(S.RAGGED_B8, n_layers=2, prefix_lens=[1500, 3333, 2048], k_keep=256),
    "xlayer_rt256": S.scaled(S.LLAMA70B_64K_XLAYER, n_layers=4, prefix_lens=[3000], layer_range=(1, 3), k_keep=256),
    "padded_max_w24": S.Workload("det_w24", 120, 2, 8, 2, 128, 24, (2500,), group_reduce="max", pool_k=5,
                                 k_keep=100, n_clusters=4),
    "logits_max_rt256": S.Workload("det_logits", 121, 1, 6, 2, 128, 40, (2100,), group_reduce="max", pool_k=3,
                                   score_mode="logits", k_keep=48),
}


def _outputs(pipe):
    outs = [pipe.scores, pipe.idx, pipe.k_out, pipe.v_out]
    for x in (pipe.page_scores, pipe.combined, pipe.agg, pipe.kv_indptr):
        if x is not None:
            outs.append(x)
    if pipe.kv_indptr is not None:
        outs.append(pipe.kv_indices[:int(pipe.kv_indptr[-1])])
    return [x.clone() for x in outs]


@pytest.mark.parametrize("name", list(CASES))
def test_two_runs_bit_equal(name, cuda):
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = CASES[name]
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    mask = inp.mask.to(cuda) if w.block_union else None
    nkv = inp.n_kvblk if w.block_union else None
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v, mask, nkv)
    first = _outputs(pipe)
    for x in (pipe.scores, pipe.k_out):
        x.fill_(float("nan") if x.dtype == torch.float32 else 0)
    pipe.idx.fill_(-5)
    pipe.run(q, k, v, mask, nkv)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    for a, b in zip(first, _outputs(pipe)):
        assert torch.equal(a, b), f"{name}: an output differs between two runs"


def test_attention_two_runs_bit_equal(cuda):
    """Attention over the selected pages, read in place: split partials merged in a fixed order."""
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200])
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v)
    qd = S.make_decode_queries(w, 1, str(cuda))
    n_sel, P = pipe.n_sel, w.page_size
    n = K.kvsel_attend_workspace_size(pipe.desc, 1, P, n_sel)
    buf = torch.zeros(n + K.WS_ALIGN, dtype=torch.uint8, device=cuda)
    off = (-buf.data_ptr()) % K.WS_ALIGN
    ws = buf[off:off + n]
    outs = []
    for _ in range(2):
        o = torch.full((1, w.n_layers, w.h_q, 1, w.head_dim), float("nan"), dtype=torch.float32, device=cuda)
        K.kvsel_attend(pipe.desc, qd, 1, k, v, None, pipe.idx, n_sel, P, n_sel, o, ws)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
