"""Guard regions around every output and the workspace: a whole pass of the path writes nothing
outside the buffers it was given (the kernels' own index arithmetic at ragged tails, partial
pages, padded row blocks and the last tile of every unit)."""

import pytest
import torch

from attention_kv_cache_gb300 import synth as S

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side; keeps the interior 256-byte aligned
FILL = 0xA5


def _guarded(shape, dtype, device):
    """A tensor of `shape` inside a byte buffer whose GUARD bytes on each side hold FILL."""
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((nbytes + 2 * GUARD,), FILL, dtype=torch.uint8, device=device)
    inner = buf[GUARD:GUARD + nbytes].view(dtype).view(shape)
    return buf, inner


def _guard_outputs(pipe, device):
    """Replaces the pipeline's output buffers and workspace by guarded ones; returns the guards."""
    guards = {}
    for name in ("scores", "page_scores", "combined", "agg", "idx", "k_out", "v_out", "kv_indptr", "kv_indices"):
        t = getattr(pipe, name, None)
        if t is None:
            continue
        buf, inner = _guarded(tuple(t.shape), t.dtype, device)
        setattr(pipe, name, inner)
        guards[name] = (buf, inner.numel() * inner.element_size())
    buf, ws = _guarded((pipe.ws_bytes,), torch.uint8, device)
    ws.zero_()
    pipe.ws = ws
    guards["ws"] = (buf, pipe.ws_bytes)
    return guards


CASES = {
    # paged: partial last page, recency pages, page maxima
    "paged": S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8200]),
    # ragged batch with the block-union CSR
    "ragged_csr": S.scaled(S.RAGGED_B8, n_layers=2, prefix_lens=[1500, 3333, 2048], k_keep=256),
    # 256 rows per unit (paired epilogue warps), cross-layer mean
    "xlayer_rt256": S.scaled(S.LLAMA70B_64K_XLAYER, n_layers=4, prefix_lens=[3001], layer_range=(1, 3), k_keep=200),
    # all-head selection with a window of 8
    "allheads_w8": S.scaled(S.LLAMA8B_32K, n_layers=2, prefix_lens=[2049], window=8, pool_type="avg",
                            head_reduce="all", k_keep=100),
}


@pytest.mark.parametrize("name", list(CASES))
def test_no_write_outside_buffers(name, cuda):
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = CASES[name]
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    guards = _guard_outputs(pipe, cuda)
    mask = nkv = None
    if w.block_union:
        mask = inp.mask.to(cuda)
        nkv = inp.n_kvblk
    pipe.run(q, k, v, mask, nkv)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(pipe.ws) == K.OK
    for key, (buf, nbytes) in guards.items():
        head = buf[:GUARD]
        tail = buf[GUARD + nbytes:]
        assert bool((head == FILL).all()), f"{name}: write before {key}"
        assert bool((tail == FILL).all()), f"{name}: write past the end of {key}"
