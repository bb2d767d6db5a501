"""Causal prefill attention on the tensor cores against the fp64 oracle, and the window scores taken
from its log-sum-exp (one pass over the prefix keys) against the oracle's scores.

Tolerances: P is rounded to bf16 before the P V product and o is stored as bf16, so
|o - oracle| <= 2^-9 * max|v| + 2^-8 * |oracle| (+1e-5); the lse is accumulated in fp32 from unrounded
probabilities, |lse - oracle| <= 1e-4; scores as everywhere (1e-3 relative + 1e-6).
"""

import numpy as np
import pytest
import torch

from attention_kv_cache_gb300 import synth as S
from oracle import kvsel_oracle as O
from tests.parity import assert_scores_close

pytestmark = pytest.mark.gpu


def _ws(K, n, cuda):
    buf = torch.zeros(n + K.WS_ALIGN, dtype=torch.uint8, device=cuda)
    off = (-buf.data_ptr()) % K.WS_ALIGN
    return buf[off:off + n]


def _run_prefill(w, cuda):
    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import desc_for, pack
    inp = S.make_inputs(w, "cpu")
    qf = [S.make_prompt_queries(w, b, "cpu") for b in range(w.batch)]
    _, k, v = pack(inp, cuda)
    q = torch.cat([x.reshape(-1) for x in qf]).to(cuda)
    o = torch.empty_like(q)
    lse = torch.empty(q.numel() // w.head_dim, dtype=torch.float32, device=cuda)
    G, W = w.group, w.window
    lse_win = torch.empty((w.batch, w.n_layers, w.h_kv, G * W), dtype=torch.float32, device=cuda)
    q_win = torch.empty((w.batch, w.n_layers, w.h_q, W, w.head_dim), dtype=torch.bfloat16, device=cuda)
    desc = desc_for(w)
    ws = _ws(K, K.kvsel_workspace_size(desc), cuda)
    K.kvsel_prefill_attention(desc, q, k, v, o, lse, lse_win, q_win, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    return inp, qf, k, v, o, lse, lse_win, q_win, desc, ws


def _check_prefill(w, inp, qf, o, lse, lse_win, q_win):
    off = 0
    for b in range(w.batch):
        N = w.prefix_lens[b] + w.window
        n = w.n_layers * w.h_q * N
        ob = o[off * w.head_dim:(off + n) * w.head_dim].view(w.n_layers, w.h_q, N, w.head_dim).double().cpu().numpy()
        lb = lse[off:off + n].view(w.n_layers, w.h_q, N).double().cpu().numpy()
        for layer in range(w.n_layers):
            qq = O._f64(qf[b][layer])
            kk = O._f64(inp.k[b][layer])
            vv = O._f64(inp.v[b][layer])
            ref_o, ref_l = O.prefill_attention(qq, kk, vv)
            bound = 2.0 ** -9 * np.abs(vv).max() + 2.0 ** -8 * np.abs(ref_o) + 1e-5
            bad = np.abs(ob[layer] - ref_o) > bound
            assert not bad.any(), f"o b{b} l{layer}: {bad.sum()} off, first {np.argwhere(bad)[0]}"
            np.testing.assert_allclose(lb[layer], ref_l, rtol=0, atol=1e-4, err_msg=f"lse b{b} l{layer}")
            L, W, G = w.prefix_lens[b], w.window, w.group
            want_win = (ref_l[:, L:] / np.log(2.0)).reshape(w.h_kv, G * W)
            np.testing.assert_allclose(lse_win[b, layer].double().cpu().numpy(), want_win, rtol=0, atol=2e-4)
            assert torch.equal(q_win[b, layer].cpu(), qf[b][layer][:, L:])
        off += n


@pytest.mark.parametrize("name,w", [
    ("one_seq_3_tiles", S.Workload("pf_small", 110, 2, 8, 2, 128, 16, (300,), k_keep=20)),
    ("eleven_tiles_g4", S.Workload("pf_long", 111, 1, 4, 1, 128, 32, (1300,), k_keep=40, n_clusters=4)),
    ("ragged_batch", S.Workload("pf_ragged", 112, 1, 4, 2, 128, 8, (200, 700), k_keep=16)),
])
def test_prefill_matches_oracle(name, w, cuda):
    inp, qf, k, v, o, lse, lse_win, q_win, desc, ws = _run_prefill(w, cuda)
    _check_prefill(w, inp, qf, o, lse, lse_win, q_win)


def test_prefill_offset_moves(cuda):
    """Logits that climb by 10 (base 2) per 128-key tile: every row's exponent offset moves at every
    tile up to its own, so O is rescaled in TMEM many times; o, lse and the window lse against the
    oracle as above."""
    from types import SimpleNamespace

    from attention_kv_cache_gb300 import kvsel as K
    from attention_kv_cache_gb300.pipeline import desc_for
    w = S.Workload("pf_climb", 113, 1, 2, 1, 128, 16, (600,), k_keep=16)
    N, d = 616, 128
    g = torch.Generator().manual_seed(13)
    u = torch.randn(d, generator=g)
    u /= u.norm()
    a = 4.0
    c = torch.arange(N, dtype=torch.float32) * (10.0 / 128) * np.log(2.0) * np.sqrt(d) / a
    kk = (c[:, None] * u[None, :] + 0.05 * torch.randn(N, d, generator=g)).to(torch.bfloat16)
    vv = torch.randn(N, d, generator=g).to(torch.bfloat16)
    qq = (a * u + 0.05 * torch.randn((1, 2, N, d), generator=g)).to(torch.bfloat16)    # [layers, h_q, N, d]
    q = qq.reshape(-1).to(cuda)
    o = torch.empty_like(q)
    lse = torch.empty(q.numel() // d, dtype=torch.float32, device=cuda)
    lse_win = torch.empty((1, 1, 1, 2 * w.window), dtype=torch.float32, device=cuda)
    q_win = torch.empty((1, 1, 2, w.window, d), dtype=torch.bfloat16, device=cuda)
    desc = desc_for(w)
    ws = _ws(K, K.kvsel_workspace_size(desc), cuda)
    K.kvsel_prefill_attention(desc, q, kk.reshape(-1).to(cuda), vv.reshape(-1).to(cuda), o, lse, lse_win, q_win, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    inp = SimpleNamespace(k=[kk.reshape(1, 1, N, d)], v=[vv.reshape(1, 1, N, d)])
    _check_prefill(w, inp, [qq], o, lse, lse_win, q_win)


def test_scores_from_prefill_lse(cuda):
    """Window scores from the prefill's lse (one pass) equal the oracle's and the two-pass scores."""
    from attention_kv_cache_gb300 import kvsel as K
    w = S.scaled(S.LLAMA8B_128K_PAGED, n_layers=2, prefix_lens=[2560], n_clusters=8)
    inp, qf, k, v, o, lse, lse_win, q_win, desc, ws = _run_prefill(w, cuda)
    L, P = w.prefix_lens[0], w.page_size
    scores = torch.empty(w.n_layers * w.h_kv * L, dtype=torch.float32, device=cuda)
    pages = torch.empty(w.n_layers * w.h_kv * (-(-L // P)), dtype=torch.float32, device=cuda)
    K.kvsel_score_from_lse(desc, q_win, k, lse_win, scores, pages, ws)
    s2 = torch.empty_like(scores)
    p2 = torch.empty_like(pages)
    K.kvsel_score(desc, q_win, k, s2, p2, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    ref = O.run_sequence(w, inp.q[0], inp.k[0], with_gather=False)
    assert_scores_close(scores.view(w.n_layers, w.h_kv, L), ref["pooled"], "scores from the prefill lse")
    assert_scores_close(pages.view(w.n_layers, w.h_kv, -1), ref["pages"], "pages from the prefill lse")
    assert_scores_close(scores.view(w.n_layers, w.h_kv, L), s2.view(w.n_layers, w.h_kv, L).double().cpu().numpy(),
                        "one pass against two passes")


def test_prefill_full_length_32k(cuda):
    """One layer of a 32K-token prompt (32768 prefix + 32 window rows: 257 query tiles, a partial last
    one, heaviest tile pairs first): o of sampled rows (the first tile, a middle tile, the last 160
    rows) and the lse of every window row against the oracle restricted to those rows; then the window
    scores from that lse against the oracle's scores of the same prompt."""
    from attention_kv_cache_gb300 import kvsel as K
    w = S.Workload("pf_32k", 114, 1, 2, 1, 128, 32, (32768,), group_reduce="sum", pool_k=7, k_keep=1024,
                   n_clusters=8)
    inp, qf, k, v, o, lse, lse_win, q_win, desc, ws = _run_prefill(w, cuda)
    N = w.prefix_lens[0] + w.window
    L, W, G = w.prefix_lens[0], w.window, w.group
    rows = list(range(0, 128)) + list(range(16384, 16512)) + list(range(N - 160, N))
    ob = o.view(w.h_q, N, w.head_dim)[:, rows].double().cpu().numpy()
    lb = lse.view(w.h_q, N)[:, rows].double().cpu().numpy()
    vv = O._f64(inp.v[0][0])
    ref_o, ref_l = O.prefill_rows(qf[0][0], inp.k[0][0], inp.v[0][0], rows)
    bound = 2.0 ** -9 * np.abs(vv).max() + 2.0 ** -8 * np.abs(ref_o) + 1e-5
    bad = np.abs(ob - ref_o) > bound
    assert not bad.any(), f"o: {bad.sum()} off, first {np.argwhere(bad)[0]}"
    np.testing.assert_allclose(lb, ref_l, rtol=0, atol=1e-4, err_msg="lse of the sampled rows")
    want_win = (ref_l[:, -W:] / np.log(2.0)).reshape(w.h_kv, G * W)
    np.testing.assert_allclose(lse_win[0, 0].double().cpu().numpy(), want_win, rtol=0, atol=2e-4)
    assert torch.equal(q_win[0, 0].cpu(), qf[0][0][:, L:])
    scores = torch.empty(w.n_layers * w.h_kv * L, dtype=torch.float32, device=cuda)
    K.kvsel_score_from_lse(desc, q_win, k, lse_win, scores, None, ws)
    torch.cuda.synchronize()
    assert K.kvsel_read_device_error(ws) == K.OK
    ref = O.run_sequence(w, inp.q[0], inp.k[0], with_gather=False)
    assert_scores_close(scores.view(w.n_layers, w.h_kv, L), ref["pooled"], "32K scores from the prefill lse")
