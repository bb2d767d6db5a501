"""Attention over the selected cache rows, read in place through a table, against the fp64 oracle.

The dense page table written by the selection (page mode), the block-union CSR of the page-table
step, and the dense cache; the same attention over the compacted copy; empty rows and block ids
outside the cache.
"""

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import synth as S
from oracle import kvsel_oracle as O

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-3, 1e-5


def _close(got, want, what):
    g = got.detach().double().cpu().numpy()
    bad = np.abs(g - want) > RTOL * np.abs(want) + ATOL
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} off; first {np.argwhere(bad)[0]}"


def _ws(K, n, cuda):
    buf = torch.zeros(n + K.WS_ALIGN, dtype=torch.uint8, device=cuda)
    off = (-buf.data_ptr()) % K.WS_ALIGN
    return buf[off:off + n]


def _ref(w, qd, kk, vv, lists, P, n_q):
    """o [n_layers, h_q, n_q, d] for one sequence; lists[layer][g] = block ids."""
    G = w.group
    n_keys = kk.shape[2]
    out = np.zeros((w.n_layers, w.h_q, n_q, w.head_dim))
    for layer in range(w.n_layers):
        for g in range(w.h_kv):
            rows = O.table_rows(lists[layer][g], P, n_keys)
            k64 = O._f64(kk[layer, g])
            v64 = O._f64(vv[layer, g])
            for h in range(g * G, (g + 1) * G):
                if len(rows):
                    out[layer, h] = O.attend(O._f64(qd[layer, h]), k64, v64, rows)
    return out


def test_attend_page_table_in_place_and_copy(cuda):
    """DELTA-style decode: attention over the pages kvsel_topk picked, in place and over the compacted copy."""
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[8208])     # L + W = 515 whole pages
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v)
    n_q = 2
    qd = S.make_decode_queries(w, n_q, "cpu")
    o = torch.empty((1, w.n_layers, w.h_q, n_q, w.head_dim), dtype=torch.float32, device=cuda)
    n_sel, P = pipe.n_sel, w.page_size
    wsb = K.kvsel_attend_workspace_size(pipe.desc, n_q, P, n_sel)
    ws = _ws(K, wsb, cuda)
    K.kvsel_attend(pipe.desc, qd.to(cuda), n_q, k, v, None, pipe.idx, n_sel, P, n_sel, o, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    idx = pipe.idx[0].cpu().numpy()
    want = _ref(w, qd[0], inp.k[0], inp.v[0], idx, P, n_q)
    _close(o[0], want, "in place")
    # the copy path: dense attention over the compacted cache (n_sel * P rows per unit)
    rows = n_sel * P
    dc = K.make_desc(n_layers=w.n_layers, h_q=w.h_q, h_kv=w.h_kv, head_dim=w.head_dim, window=w.window,
                     prefix_lens=[rows - w.window])
    oc = torch.empty_like(o)
    wsc = _ws(K, K.kvsel_attend_workspace_size(dc, n_q, P, n_sel), cuda)
    K.kvsel_attend(dc, qd.to(cuda), n_q, pipe.k_out.reshape(-1), pipe.v_out.reshape(-1), None, None, 0, P, n_sel,
                   oc, wsc)
    torch.cuda.synchronize()
    _close(oc[0], want, "compacted copy")


def test_attend_block_union_csr(cuda):
    """CompactAttention execution: attention over each group's block list T[b, g] (CSR), ragged batch."""
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = S.scaled(S.RAGGED_B8, n_layers=2, prefix_lens=[1500, 3333, 2048], k_keep=256, mask_density=0.25)
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v, inp.mask.to(cuda), inp.n_kvblk)
    n_q = 1
    qd = S.make_decode_queries(w, n_q, "cpu")
    o = torch.empty((w.batch, w.n_layers, w.h_q, n_q, w.head_dim), dtype=torch.float32, device=cuda)
    ws = _ws(K, K.kvsel_attend_workspace_size(pipe.desc, n_q, w.block, pipe.n_kvblk_max), cuda)
    K.kvsel_attend(pipe.desc, qd.to(cuda), n_q, k, v, pipe.kv_indptr, pipe.kv_indices, 0, w.block,
                   pipe.n_kvblk_max, o, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    M = inp.mask.numpy()
    for b in range(w.batch):
        lists = [O.block_union(M[b, layer], w.h_kv, inp.n_kvblk[b]) for layer in range(w.n_layers)]
        _close(o[b], _ref(w, qd[b], inp.k[b], inp.v[b], lists, w.block, n_q), f"csr b{b}")


def test_attend_dense_cache_and_edges(cuda):
    """No table: every cache row; empty CSR rows give 0; a block id outside the cache is skipped and reported."""
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import pack
    w = S.Workload("attend_edge", 101, 1, 8, 2, 64, 8, (777,), k_keep=10)
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    desc = K.make_desc(n_layers=1, h_q=8, h_kv=2, head_dim=64, window=8, prefix_lens=[777])
    n_q = 3
    qd = S.make_decode_queries(w, n_q, "cpu")
    n_keys = 785
    P = 16
    nb = -(-n_keys // P)
    o = torch.empty((1, 1, 8, n_q, 64), dtype=torch.float32, device=cuda)
    ws = _ws(K, K.kvsel_attend_workspace_size(desc, n_q, P, nb), cuda)
    K.kvsel_attend(desc, qd.to(cuda), n_q, k, v, None, None, 0, P, nb, o, ws)
    torch.cuda.synchronize()
    _close(o[0], _ref(w, qd[0], inp.k[0], inp.v[0], [[np.arange(nb)] * 2], P, n_q), "dense cache")
    # CSR: group 0 selects nothing, group 1 selects blocks 3, 0, 49 (the last, partial) and 99 (outside)
    indptr = torch.tensor([0, 0, 4], dtype=torch.int32, device=cuda)
    indices = torch.tensor([3, 0, 49, 99], dtype=torch.int32, device=cuda)
    K.kvsel_attend(desc, qd.to(cuda), n_q, k, v, indptr, indices, 0, P, 4, o, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.ERR_DEVICE
    assert torch.all(o[0, 0, :4] == 0)
    want = _ref(w, qd[0], inp.k[0], inp.v[0], [[np.zeros(0, np.int64), np.array([3, 0, 49])]], P, n_q)
    _close(o[0, 0, 4:], want[0, 4:], "csr with an empty row")


@pytest.mark.parametrize("h_q,h_kv,n_q,d", [(2, 2, 1, 128), (6, 2, 1, 128), (6, 2, 2, 64), (8, 1, 1, 128)])
def test_attend_group_shapes(h_q, h_kv, n_q, d, cuda):
    """Query rows per table row R = (h_q / h_kv) * n_q of 1, 3, 6 and 8 (padded decode kernels) over a page list."""
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import pack
    w = S.Workload("attend_shape", 102, 2, h_q, h_kv, d, 4, (1001,), k_keep=10)
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    desc = K.make_desc(n_layers=2, h_q=h_q, h_kv=h_kv, head_dim=d, window=4, prefix_lens=[1001])
    P = 8
    g = torch.Generator().manual_seed(h_q * 100 + n_q)
    n_per = 40
    idx = torch.stack([torch.randperm(126, generator=g)[:n_per] for _ in range(2 * h_kv)]).int()   # 126 pages
    qd = S.make_decode_queries(w, n_q, "cpu")
    o = torch.empty((1, 2, h_q, n_q, d), dtype=torch.float32, device=cuda)
    ws = _ws(K, K.kvsel_attend_workspace_size(desc, n_q, P, n_per), cuda)
    K.kvsel_attend(desc, qd.to(cuda), n_q, k, v, None, idx.to(cuda), n_per, P, n_per, o, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    lists = idx.view(2, h_kv, n_per).numpy()
    _close(o[0], _ref(w, qd[0], inp.k[0], inp.v[0], lists, P, n_q), f"R={h_q // h_kv * n_q}")


def _climbing(n_keys, d, slope2, a, seed):
    """Unit direction u, K rows c_t u (+ small noise) whose logit against the query a u grows by slope2
    (base 2) per key, and random V rows: (u, k [n_keys, d] bf16, v [n_keys, d] bf16)."""
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(d, generator=g)
    u /= u.norm()
    c = torch.arange(n_keys, dtype=torch.float32) * slope2 * np.log(2.0) * np.sqrt(d) / a
    k = (c[:, None] * u[None, :] + 0.05 * torch.randn(n_keys, d, generator=g)).to(torch.bfloat16)
    v = torch.randn(n_keys, d, generator=g).to(torch.bfloat16)
    return u, k, v


@pytest.mark.parametrize("n_q", [1, 3])
def test_attend_offset_moves(n_q, cuda):
    """Logits that climb by 12 (base 2) per 128 keys along the cache: within every split the exponent
    offset moves many times (O and l rescaled), and the splits' offsets differ by far more than 2^8 in
    the merge.  R = 4 (tensor-core warp kernel) and R = 12 (block kernel)."""
    from attention_kv_cache_gb300 import kvsel as K
    h_q, d, L, W, P = 4, 128, 3000, 8, 16
    n_keys = L + W
    w = S.Workload("attend_climb", 103, 1, h_q, 1, d, W, (L,), k_keep=10)
    u, kk, vv = _climbing(n_keys, d, 12.0 / 128, 4.0, seed=7 + n_q)
    g = torch.Generator().manual_seed(11)
    qd = (4.0 * u + 0.05 * torch.randn((1, 1, h_q, n_q, d), generator=g)).to(torch.bfloat16)
    desc = K.make_desc(n_layers=1, h_q=h_q, h_kv=1, head_dim=d, window=W, prefix_lens=[L])
    nb = -(-n_keys // P)
    o = torch.empty((1, 1, h_q, n_q, d), dtype=torch.float32, device=cuda)
    ws = _ws(K, K.kvsel_attend_workspace_size(desc, n_q, P, nb), cuda)
    K.kvsel_attend(desc, qd.to(cuda), n_q, kk.reshape(-1).to(cuda), vv.reshape(-1).to(cuda), None, None, 0, P, nb,
                   o, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    want = _ref(w, qd[0], kk[None, None], vv[None, None], [[np.arange(nb)]], P, n_q)
    _close(o[0], want, f"climbing logits R={h_q * n_q}")


def test_attend_full_size_page_table_128k(cuda):
    """One layer of the 128K paged workload at full length: the selection's 134 pages per (KV head) row
    (128 chosen + 4 recent + 2 window pages of 16 rows) attended in place, against the oracle."""
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import Pipeline, pack
    w = S.scaled(S.LLAMA8B_128K_PAGED, n_layers=1)
    inp = S.make_inputs(w, "cpu")
    q, k, v = pack(inp, cuda)
    pipe = Pipeline(w, cuda)
    pipe.run(q, k, v)
    n_q = 1
    qd = S.make_decode_queries(w, n_q, "cpu")
    o = torch.empty((1, w.n_layers, w.h_q, n_q, w.head_dim), dtype=torch.float32, device=cuda)
    n_sel, P = pipe.n_sel, w.page_size
    assert n_sel == 134
    ws = _ws(K, K.kvsel_attend_workspace_size(pipe.desc, n_q, P, n_sel), cuda)
    K.kvsel_attend(pipe.desc, qd.to(cuda), n_q, k, v, None, pipe.idx, n_sel, P, n_sel, o, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    idx = pipe.idx[0].cpu().numpy()
    _close(o[0], _ref(w, qd[0], inp.k[0], inp.v[0], idx, P, n_q), "128K page table in place")
