"""The whole path captured in a CUDA graph and replayed.

No entry point of a step synchronises, allocates or copies through the host, so a step can be
captured once (torch.cuda.graph, global capture mode) and replayed: each replay must write exactly
the bits an eager run writes, and must read the live input buffers (new values in the same tensors
give the eager result for the new values).  Covered: page mode, a ragged batch with the block-union
page table, the cross-layer mean over 256-row units, prefix lengths read on the device, and the
gather reading V from mapped pinned host memory.
"""

import pytest
import torch

from attention_kv_cache_gb300 import kvsel as K
from attention_kv_cache_gb300 import synth as S

pytestmark = pytest.mark.gpu

CASES = {
    "paged_max": S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200]),
    "ragged_csr": S.scaled(S.RAGGED_B8, n_layers=2, prefix_lens=[1500, 3333, 2048], k_keep=256),
    "xlayer_rt256": S.scaled(S.LLAMA70B_64K_XLAYER, n_layers=4, prefix_lens=[3000], layer_range=(1, 3), k_keep=256),
}


def _bits(x):
    """The tensor's bits (buffers sized for a length bound keep NaN fill past the real lengths)."""
    if x.dtype == torch.float32:
        return x.view(torch.int32)
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16)
    return x


def _outputs(pipe):
    outs = [pipe.scores, pipe.idx, pipe.k_out, pipe.v_out]
    for x in (pipe.page_scores, pipe.combined, pipe.agg, pipe.kv_indptr):
        if x is not None:
            outs.append(x)
    if pipe.kv_indptr is not None:
        outs.append(pipe.kv_indices[:int(pipe.kv_indptr[-1])])
    return [_bits(x).clone() for x in outs]


def _clear(pipe):
    for x in (pipe.scores, pipe.k_out, pipe.v_out):
        x.fill_(float("nan") if x.dtype == torch.float32 else 0)
    pipe.idx.fill_(-5)


def _capture(fn):
    """Warm up on a side stream, then capture fn() into a graph (torch's default: global mode)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _replay_matches_eager(pipe, run, refill):
    _clear(pipe)
    run()
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    eager = _outputs(pipe)
    g = _capture(run)
    for _ in range(2):
        _clear(pipe)
        g.replay()
        torch.cuda.synchronize()
        assert K.kvsel_read_device_error(pipe.ws) == K.OK
        for a, b in zip(eager, _outputs(pipe)):
            assert torch.equal(a, b), "a replay differs from the eager run"
    # the graph reads the buffers as they are at replay time
    refill()
    _clear(pipe)
    run()
    torch.cuda.synchronize()
    eager2 = _outputs(pipe)
    assert not torch.equal(eager[0], eager2[0])
    _clear(pipe)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager2, _outputs(pipe)):
        assert torch.equal(a, b), "a replay after new inputs differs from the eager run on them"


@pytest.mark.parametrize("name", list(CASES))
def test_step_replays_bit_equal(name, cuda):
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = CASES[name]
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    mask = inp.mask.to(cuda) if w.block_union else None
    nkv = inp.n_kvblk if w.block_union else None
    pipe = Pipeline(w, cuda)
    q2 = torch.flip(q, dims=[-2]).contiguous()          # another window: the rows in reverse order

    def refill():
        q.copy_(q2)

    _replay_matches_eager(pipe, lambda: pipe.run(q, k, v, mask, nkv), refill)


def test_device_lengths_and_host_values_replay(cuda):
    """Lengths read on the device and V read from pinned host memory, inside the captured step."""
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = S.scaled(S.LLAMA8B_32K, n_layers=2, prefix_lens=[4000, 2500])
    inp = S.make_inputs(w, "cpu")
    q, k0, v0 = pack(inp, cuda)
    lens = torch.tensor(w.prefix_lens, dtype=torch.int64, device=cuda)
    len_max = 4100
    pipe = Pipeline(w, cuda, lens_dev=lens, len_max=len_max)
    # K and V packed by the real lengths inside buffers with room for every sequence at the bound
    cap = w.batch * w.n_layers * w.h_kv * (len_max + w.window) * w.head_dim
    k = torch.zeros(cap, dtype=torch.bfloat16, device=cuda)
    k[:k0.numel()] = k0
    vh = torch.zeros(cap, dtype=torch.bfloat16).pin_memory()
    vh[:v0.numel()] = v0.cpu()
    q2 = torch.flip(q, dims=[-2]).contiguous()

    def refill():
        q.copy_(q2)

    _replay_matches_eager(pipe, lambda: pipe.run(q, k, vh), refill)
