"""Pins for the fp64 oracle: checks against facts fixed outside the oracle itself.

Each ``check_*`` takes the oracle module (or a mutated copy of it) and raises
AssertionError when the oracle disagrees with:

* an independent library routine computing the same quantity
  (torch's scaled_dot_product_attention with identity values returns the
  masked softmax probabilities, and its ``enable_gqa`` fixes the query-head
  to KV-head map; scipy's softmax for the one-row case);
* closed forms (identical keys; a hand-worked 4-key example);
* invariants (softmax rows sum to one, so each head's column mass over all
  visible columns is exactly W; L1-normalised scores sum to one);
* brute force on tiny inputs (subset enumeration for top-k with ties, loop
  definitions of pooling, page reduction and the block unions).

``tests/test_oracle_pins.py`` runs them on the oracle; ``tests/test_oracle_mutants.py``
plants plausible mistakes in copies of the oracle and checks that some pin fails.
"""

from __future__ import annotations

import itertools
import math

import numpy as np
import torch


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_values(a: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 and back, so inputs look like the workloads'."""
    return torch.from_numpy(a).to(torch.bfloat16).double().numpy()


# --------------------------------------------------------------------------- scoring pins

def check_probs_match_sdpa(o):
    """Group scores and probabilities equal torch SDPA's attention weights (identity values, GQA map)."""
    rng = _rng(1)
    Hq, Hkv, W, L, d = 6, 2, 5, 13, 8
    G = Hq // Hkv
    q = _bf16_values(rng.standard_normal((Hq, W, d)) * 1.7)
    k = _bf16_values(rng.standard_normal((Hkv, L + W, d)) * 1.3)
    N = L + W
    # attention weights = SDPA(q, k, V = I): output row r is the probability row of query r
    vis = torch.zeros((W, N), dtype=torch.bool)
    for j in range(W):
        vis[j, : L + j + 1] = True            # window row j at position L + j sees keys 0 .. L + j
    eye = torch.eye(N, dtype=torch.float64).expand(Hkv, N, N)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], eye[None],
        attn_mask=vis, enable_gqa=True)[0].numpy()           # [Hq, W, N]
    for mode in ("sum", "max"):
        for g in range(Hkv):
            s = o.score_unit(q, k, g, G, L, mode)
            heads = ref[g * G:(g + 1) * G, :, :L].sum(axis=1)     # column mass per head
            want = heads.sum(axis=0) if mode == "sum" else heads.max(axis=0)
            np.testing.assert_allclose(s, want, rtol=1e-12, atol=1e-15)
    for g in range(Hkv):
        p = o.window_probs(q[g * G:(g + 1) * G], k[g], L)
        np.testing.assert_allclose(p, ref[g * G:(g + 1) * G], rtol=1e-12, atol=1e-15)


def check_row_mass_invariant(o):
    """Each softmax row sums to one, so a head's mass over all visible columns is W, and the prefix part is below it."""
    rng = _rng(2)
    G, W, L, d = 3, 7, 40, 16
    q = rng.standard_normal((G, W, d)) * 2.0
    k = rng.standard_normal((L + W, d))
    p = o.window_probs(q, k, L)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p[:, np.arange(W)[:, None] < np.arange(L + W)[None, :] - L] == 0.0)
    c = o.column_mass(p, L)
    assert c.shape == (G, L)
    total = c.sum(axis=1) + p[:, :, L:].sum(axis=(1, 2))
    np.testing.assert_allclose(total, W, rtol=0, atol=1e-10)
    s = o.group_reduce(c, "sum")
    assert s.sum() <= G * W + 1e-9


def check_identical_keys_closed_form(o):
    """All keys equal: row j has L + j + 1 equal logits, so c[h, t] = sum_j 1 / (L + j + 1) for every prefix t."""
    rng = _rng(3)
    G, W, L, d = 2, 6, 30, 8
    q = rng.standard_normal((G, W, d))
    k = np.tile(rng.standard_normal((1, d)), (L + W, 1))
    want = sum(1.0 / (L + j + 1) for j in range(W))
    for mode, factor in (("sum", G), ("max", 1)):
        s = o.group_scores(q, k, L, mode)
        np.testing.assert_allclose(s, factor * want, rtol=1e-12)
    u = o.max_pool(o.group_scores(q, k, L, "sum"), 7)
    np.testing.assert_allclose(u, G * want, rtol=1e-12)
    # ties everywhere: the first k positions win, then the window follows
    idx = o.select_tokens(u, 5, L, W)
    assert list(idx) == list(range(5)) + list(range(L, L + W))


def check_hand_worked_example(o):
    """d = 4 (scale 1/2), L = 2, W = 2, one head.

    q_0 = (2 ln 2, 0, 0, 0), q_1 = 0; k_0 = (1, 0, 0, 0), k_1 = k_2 = k_3 = 0.
    Row 0 sees keys 0..2 with logits (ln 2, 0, 0): p = (2, 1, 1) / 4.
    Row 1 sees keys 0..3, all logits 0: p = 1/4 each.
    Column mass over the prefix: c_0 = 1/2 + 1/4 = 3/4, c_1 = 1/4 + 1/4 = 1/2.
    """
    q = np.zeros((1, 2, 4)); q[0, 0, 0] = 2.0 * math.log(2.0)
    k = np.zeros((4, 4)); k[0, 0] = 1.0
    p = o.window_probs(q, k, 2)
    np.testing.assert_allclose(p[0, 0], [0.5, 0.25, 0.25, 0.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(p[0, 1], [0.25] * 4, rtol=0, atol=1e-15)
    np.testing.assert_allclose(o.group_scores(q, k, 2, "sum"), [0.75, 0.5], rtol=0, atol=1e-15)


def check_one_row_textbook(o):
    """W = 1, G = 1, no pooling: the scores are one softmax row over L + 1 keys (scipy), first L entries."""
    from scipy.special import softmax
    rng = _rng(4)
    L, d = 25, 12
    q = rng.standard_normal((1, 1, d)) * 3.0
    k = rng.standard_normal((L + 1, d))
    z = np.array([sum(q[0, 0, c] * k[t, c] for c in range(d)) / math.sqrt(d) for t in range(L + 1)])
    want = softmax(z)[:L]
    np.testing.assert_allclose(o.group_scores(q, k, L, "sum"), want, rtol=1e-12)
    np.testing.assert_allclose(o.group_scores(q, k, L, "max"), want, rtol=1e-12)


def check_planted_key_first(o):
    """A prefix key 8 sqrt(d) along the mean window-query direction ranks first and is always selected."""
    rng = _rng(5)
    G, W, L, d = 4, 8, 200, 32
    q = rng.standard_normal((G, W, d))
    k = rng.standard_normal((L + W, d))
    u = q.reshape(-1, d).mean(axis=0)
    u /= np.linalg.norm(u)
    for pos in (0, 77, L - 1):
        kk = k.copy()
        kk[pos] = 8.0 * math.sqrt(d) * u
        for mode in ("sum", "max"):
            s = o.group_scores(q, kk, L, mode)
            assert int(np.argmax(s)) == pos
            assert o.rank(s)[0] == pos
            idx = o.select_tokens(o.max_pool(s, 1), 1, L, W)
            assert idx[0] == pos


# --------------------------------------------------------------------------- pooling / pages

def _pool_loop(s, k):
    r = (k - 1) // 2
    n = len(s)
    return np.array([max(s[max(0, t - r):min(n, t + r + 1)]) for t in range(n)])


def check_pool_definition(o):
    """Max-pool equals its loop definition; a single spike widens to exactly 2r + 1 positions (clipped at the ends)."""
    rng = _rng(6)
    for n in (1, 2, 3, 7, 8, 50):
        s = rng.random(n)
        for kk in (1, 3, 7, 9):
            np.testing.assert_array_equal(o.max_pool(s, kk), _pool_loop(s, kk))
    for pos in (0, 2, 10, 19):
        s = np.zeros(20); s[pos] = 1.0
        u = o.max_pool(s, 7)
        assert list(np.nonzero(u)[0]) == list(range(max(0, pos - 3), min(20, pos + 4)))
    s = rng.random((3, 4, 33))
    np.testing.assert_array_equal(o.max_pool(s, 7)[1, 2], _pool_loop(s[1, 2], 7))


def check_page_reduce_definition(o):
    """Page max / sum over P consecutive tokens, the last page partial."""
    rng = _rng(7)
    for n in (16, 17, 31, 48, 5):
        u = rng.random(n)
        P = 16
        n_pages = -(-n // P)
        want_max = [max(u[p * P:min(n, (p + 1) * P)]) for p in range(n_pages)]
        want_sum = [sum(u[p * P:min(n, (p + 1) * P)]) for p in range(n_pages)]
        np.testing.assert_array_equal(o.page_reduce(u, P, "max"), want_max)
        np.testing.assert_allclose(o.page_reduce(u, P, "sum"), want_sum, rtol=1e-15)


# --------------------------------------------------------------------------- selection

def _brute_topk(scores, k):
    """Best k-subset: max score sum, then the lexicographically smallest ascending index tuple."""
    best = None
    for sub in itertools.combinations(range(len(scores)), k):
        key = (-sum(scores[list(sub)]), sub)
        if best is None or key < best:
            best = key
    return list(best[1])


def check_topk_brute_force(o):
    """Sort-based top-k with ties to the lower index equals subset enumeration (exact sums on 1/8 levels)."""
    rng = _rng(8)
    for trial in range(40):
        n = int(rng.integers(1, 12))
        s = rng.integers(0, 4, n) * 0.125
        for k in range(1, min(n, 4) + 1):
            got = list(o.select_tokens(s, k, n, 0))
            assert got == _brute_topk(s, k), (s, k, got)
    # the window is appended after the ascending selection
    s = np.array([0.0, 3.0, 1.0, 3.0, 2.0])
    assert list(o.select_tokens(s, 2, 5, 3)) == [1, 3, 5, 6, 7]


def check_page_selection_rule(o):
    """Recency pages always kept, the top k of the other prefix pages by brute force, then window pages."""
    rng = _rng(9)
    P, W = 4, 8
    for trial in range(30):
        L = int(rng.integers(9, 40))
        n_pages = -(-L // P)
        n_recent = int(rng.integers(1, 3))
        cand = n_pages - n_recent
        k = int(rng.integers(1, min(cand, 3) + 1))
        U = rng.integers(0, 3, n_pages) * 0.5
        got = list(o.select_pages(U, k, n_recent, L, W, P))
        top = _brute_topk(U[:cand], k)
        want = sorted(top + list(range(cand, n_pages)))
        wp = list(range(n_pages, -(-(L + W) // P)))
        assert got == want + wp, (L, n_recent, k, U, got)
        if L % P == 0:
            assert len(got) == k + n_recent + W // P


def check_gather(o):
    rng = _rng(10)
    x = rng.standard_normal((37, 5))
    idx = np.array([0, 3, 36])
    np.testing.assert_array_equal(o.gather_rows(x, idx), x[[0, 3, 36]])
    pg = o.gather_rows(x, np.array([1, 9]), 4)
    np.testing.assert_array_equal(pg[:4], x[4:8])
    np.testing.assert_array_equal(pg[4], x[36])
    np.testing.assert_array_equal(pg[5:], 0.0)


# --------------------------------------------------------------------------- cross-layer

def check_l1_cross_layer(o):
    """L1-normalised rows sum to one; the layer mean sums to one; scaling one layer changes nothing."""
    rng = _rng(11)
    s = rng.random((6, 3, 50)) * rng.random((6, 3, 1)) * 10
    S = o.cross_layer_mean(s, 1, 4)
    np.testing.assert_allclose(S.sum(axis=-1), 1.0, rtol=1e-13)
    s2 = s.copy(); s2[2] *= 37.0; s2[0] *= 5.0; s2[5] *= 0.01
    np.testing.assert_allclose(o.cross_layer_mean(s2, 1, 4), S, rtol=1e-13)
    # a layer outside the range does not matter; a layer inside it does
    s3 = s.copy(); s3[5] = rng.random((3, 50))
    np.testing.assert_allclose(o.cross_layer_mean(s3, 1, 4), S, rtol=1e-13)
    s4 = s.copy(); s4[4] = rng.random((3, 50))
    assert np.abs(o.cross_layer_mean(s4, 1, 4) - S).max() > 1e-6
    # with identical normalised layers the mean is that layer
    one = rng.random((1, 2, 9))
    same = np.concatenate([one * c for c in (1.0, 2.0, 3.0)])
    np.testing.assert_allclose(o.cross_layer_mean(same, 0, 2), one[0] / one[0].sum(-1, keepdims=True), rtol=1e-13)


# --------------------------------------------------------------------------- block union

def check_block_union(o):
    """CSR equals the OR over (Q block, head in group) by array reduction; minimal and complete."""
    rng = _rng(12)
    B, Lyr, Hq, Hkv, nq, nmax = 3, 2, 8, 2, 5, 23
    n_kv = [23, 9, 17]
    M = (rng.random((B, Lyr, Hq, nq, nmax)) < 0.08).astype(np.uint8)
    indptr, indices = o.block_union_csr(M, Hkv, n_kv)
    G = Hq // Hkv
    row = 0
    for b in range(B):
        for layer in range(Lyr):
            for g in range(Hkv):
                block = M[b, layer, g * G:(g + 1) * G, :, :n_kv[b]]
                want = np.nonzero(block.any(axis=(0, 1)))[0]
                got = indices[indptr[row]:indptr[row + 1]]
                np.testing.assert_array_equal(got, want)
                for j in got:           # minimal: every listed block was selected by some (h, i)
                    assert block[:, :, j].any()
                for h, i, j in zip(*np.nonzero(block)):   # complete: every selected block is listed
                    assert j in got
                assert np.all(np.diff(got) > 0)
                row += 1
    assert row == B * Lyr * Hkv and indptr[-1] == len(indices)


# --------------------------------------------------------------------------- scoring variants

def _sdpa_probs(q, k, L, W):
    """Window-row attention weights from torch SDPA with identity values: [Hq, W, L + W]."""
    N = L + W
    Hkv = k.shape[0]
    vis = torch.zeros((W, N), dtype=torch.bool)
    for j in range(W):
        vis[j, : L + j + 1] = True
    eye = torch.eye(N, dtype=torch.float64).expand(Hkv, N, N)
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], eye[None], attn_mask=vis, enable_gqa=True)[0].numpy()


def check_logits_mode_sdpa_log_ratios(o):
    """Pre-softmax scores: per row, z[t] - z[0] = log p[t] - log p[0] with p from torch SDPA (the GQA map and
    scale included), summed over the window rows; the level is fixed by a hand-worked logit."""
    rng = _rng(13)
    Hq, Hkv, W, L, d = 6, 2, 3, 11, 8
    G = Hq // Hkv
    q = _bf16_values(rng.standard_normal((Hq, W, d)))
    k = _bf16_values(rng.standard_normal((Hkv, L + W, d)))
    p = _sdpa_probs(q, k, L, W)
    lr = np.log(p[:, :, :L]) - np.log(p[:, :, :1])              # [Hq, W, L]
    for g in range(Hkv):
        heads = lr[g * G:(g + 1) * G].sum(axis=1)                # [G, L]
        for mode in ("sum", "max"):
            s = o.score_unit(q, k, g, G, L, mode, softmax=False)
            want_diff = heads.sum(axis=0) if mode == "sum" else None
            if mode == "sum":
                np.testing.assert_allclose(s - s[0], want_diff, atol=1e-10)
            else:
                # each head's logit mass differs from its own first column by the SDPA log ratios
                c = np.stack([o.score_unit(q[g * G + h:g * G + h + 1], k[g:g + 1], 0, 1, L, "sum", softmax=False)
                              for h in range(G)])
                np.testing.assert_allclose(c - c[:, :1], heads, atol=1e-10)
                np.testing.assert_allclose(s, c.max(axis=0), rtol=0, atol=0)
    # level: d = 4, q = (1, 1, 1, 1), k_t = (1, 0, 0, 0) gives z = 1/2; W = 2 equal rows give 1
    q1 = np.ones((1, 2, 4))
    k1 = np.zeros((5, 4)); k1[:, 0] = 1.0
    np.testing.assert_allclose(o.group_scores(q1, k1, 3, "sum", softmax=False), [1.0, 1.0, 1.0], rtol=1e-15)


def check_mean_reduce_and_head_sum(o):
    """'mean' = the group's probabilities averaged over its G*W rows; the sum over all KV heads of the
    group sums is the sum over every query head's rows (torch SDPA)."""
    rng = _rng(14)
    Hq, Hkv, W, L, d = 8, 2, 4, 9, 8
    G = Hq // Hkv
    q = _bf16_values(rng.standard_normal((Hq, W, d)) * 1.5)
    k = _bf16_values(rng.standard_normal((Hkv, L + W, d)))
    p = _sdpa_probs(q, k, L, W)[:, :, :L]
    for g in range(Hkv):
        np.testing.assert_allclose(o.score_unit(q, k, g, G, L, "mean"), p[g * G:(g + 1) * G].mean(axis=(0, 1)),
                                   rtol=1e-12)
    per_group = np.stack([o.score_unit(q, k, g, G, L, "sum") for g in range(Hkv)])
    np.testing.assert_allclose(o.head_sum(per_group), p.sum(axis=(0, 1)), rtol=1e-12)
    np.testing.assert_allclose(o.head_sum(per_group[None])[0], p.sum(axis=(0, 1)), rtol=1e-12)


def _avg_loop(s, k):
    r = (k - 1) // 2
    n = len(s)
    return np.array([np.mean(s[max(0, t - r):min(n, t + r + 1)]) for t in range(n)])


def check_avg_pool_definition(o):
    """Average pool equals its loop definition (in-range neighbours counted); constants stay constant;
    a unit spike spreads as 1 / (number of in-range neighbours)."""
    rng = _rng(15)
    for n in (1, 2, 3, 7, 8, 41):
        s = rng.random(n)
        for kk in (1, 3, 7, 9):
            np.testing.assert_allclose(o.avg_pool(s, kk), _avg_loop(s, kk), rtol=1e-14)
            np.testing.assert_allclose(o.pool(s, kk, "avg"), _avg_loop(s, kk), rtol=1e-14)
        np.testing.assert_allclose(o.avg_pool(np.full(n, 2.5), 7), 2.5, rtol=1e-15)
    s = np.zeros(20); s[0] = 1.0
    np.testing.assert_allclose(o.avg_pool(s, 7)[:5], [1 / 4, 1 / 5, 1 / 6, 1 / 7, 0.0], rtol=1e-15)
    x = rng.random((2, 3, 17))
    np.testing.assert_allclose(o.avg_pool(x, 5)[1, 2], _avg_loop(x[1, 2], 5), rtol=1e-14)
    np.testing.assert_array_equal(o.pool(x, 5, "max"), o.max_pool(x, 5))


def check_layer_max_and_keep_count(o):
    """Token-wise max over an inclusive layer range by brute force; keep counts round half up."""
    rng = _rng(16)
    s = rng.random((7, 3, 13))
    m = o.layer_max(s, 2, 5)
    for i in range(3):
        for t in range(13):
            assert m[i, t] == max(s[l, i, t] for l in range(2, 6))
    assert np.all(m >= s[2:6]) and not np.all(m >= s[6])
    table = {(0.2, 32768): 6554, (0.1, 30): 3, (0.25, 10): 3, (0.15, 10): 2, (1.0, 7): 7, (0.0, 5): 0,
             (0.5, 1): 1, (0.4, 3): 1, (0.1, 32768): 3277}
    for (r, L), want in table.items():
        assert o.keep_count(r, L) == want, (r, L, o.keep_count(r, L))


def check_claa_max_buffer(o):
    """CLAA: a key that only one buffered layer attends to strongly enters the prune index (token-wise
    max, not a mean), a key attended only just before the buffer does not, and every layer's own
    index is the top-k of its pooled all-head window score."""
    rng = _rng(17)
    n_layers, Hq, Hkv, W, L, d = 8, 4, 2, 2, 40, 16
    G = Hq // Hkv
    q = rng.standard_normal((n_layers, Hq, W, d))
    k = rng.standard_normal((n_layers, Hkv, L + W, d)) * 0.3
    defer, lp, nbuf = 2, 6, 3                       # buffer = layers 4, 5, 6
    u = q.sum(axis=(1, 2))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    for g in range(Hkv):
        k[5, g, 10] = 6.0 * np.sqrt(d) * u[5]      # inside the buffer, one layer only
        k[3, g, 30] = 6.0 * np.sqrt(d) * u[3]      # a layer before the buffer
    res = o.claa_sequence(q, k, L, W, G, Hkv, defer, lp, nbuf, keep_rate=0.1, pool_k=1)
    assert res["buffer"] == (4, 6) and res["k"] == 4
    assert 10 in res["prune_idx"] and 30 not in res["prune_idx"]
    assert 30 in res["layer_idx"][3] and 10 in res["layer_idx"][5]
    for l in range(defer, lp + 1):
        s = sum(o.score_unit(q[l], k[l], g, G, L, "sum") for g in range(Hkv))
        np.testing.assert_allclose(res["layer_scores"][l], s, rtol=1e-13)
    # with identical layers the aggregate is that layer and the prune index is its index
    q2 = np.repeat(q[:1], n_layers, axis=0)
    k2 = np.repeat(k[:1], n_layers, axis=0)
    r2 = o.claa_sequence(q2, k2, L, W, G, Hkv, 1, 5, 4, keep_rate=0.2)
    np.testing.assert_array_equal(r2["prune_idx"], r2["layer_idx"][5])
    assert r2["buffer"] == (2, 5)
    # the buffer never reaches below the deferred layers
    assert o.claa_sequence(q, k, L, W, G, Hkv, 5, 6, 4, keep_rate=0.1)["buffer"] == (5, 6)


# --------------------------------------------------------------------------- attention over a table

def check_table_attention_sdpa(o):
    """Attention over table rows equals torch SDPA on the gathered rows (scale, softmax, weighted V);
    identical keys give the plain mean of the V rows; block rows past the cache end do not exist."""
    rng = _rng(18)
    N, d, R, P = 70, 16, 5, 8
    k = _bf16_values(rng.standard_normal((N, d)) * 1.3)
    v = _bf16_values(rng.standard_normal((N, d)))
    q = _bf16_values(rng.standard_normal((R, d)))
    blocks = np.array([8, 0, 3, 5])                     # block 8 covers rows 64..71: only 64..69 exist
    rows = o.table_rows(blocks, P, N)
    assert list(rows) == list(range(64, 70)) + list(range(0, 8)) + list(range(24, 32)) + list(range(40, 48))
    got = o.attend(q, k, v, rows)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(k[rows])[None, None], torch.from_numpy(v[rows])[None, None]
    )[0, 0].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
    same = np.repeat(k[:1], N, axis=0)
    np.testing.assert_allclose(o.attend(q, same, v, rows), np.repeat(v[rows].mean(axis=0, keepdims=True), R, 0),
                               rtol=1e-12)
    # the row order of the table does not matter
    np.testing.assert_allclose(o.attend(q, k, v, rows[::-1].copy()), got, rtol=1e-12)


def check_prefill_attention_sdpa(o):
    """Causal prefill attention equals torch SDPA (is_causal, enable_gqa); its lse reproduces the row
    weights (exp(z - lse) sums to one) and the window rows' softmax of the window scoring."""
    rng = _rng(19)
    Hq, Hkv, N, d = 4, 2, 23, 8
    q = _bf16_values(rng.standard_normal((Hq, N, d)) * 1.4)
    k = _bf16_values(rng.standard_normal((Hkv, N, d)))
    v = _bf16_values(rng.standard_normal((Hkv, N, d)))
    out, lse = o.prefill_attention(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None], is_causal=True,
        enable_gqa=True)[0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    G = Hq // Hkv
    for h in range(Hq):
        z = (q[h] @ k[h // G].T) / np.sqrt(d)
        for i in range(N):
            np.testing.assert_allclose(np.exp(z[i, :i + 1] - lse[h, i]).sum(), 1.0, rtol=1e-13)
    # any subset of rows, computed alone, equals those rows of the whole prompt (and SDPA's causal output)
    rows = [0, 1, 7, 13, N - 1]
    o_r, l_r = o.prefill_rows(q, k, v, rows)
    np.testing.assert_allclose(o_r, ref[:, rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l_r, lse[:, rows], rtol=1e-13, atol=1e-13)
    # the last W rows are the observation window: their probabilities are the window softmax
    W = 5
    L = N - W
    p = o.window_probs(q[:G, L:], k[0], L)
    for hl in range(G):
        for j in range(W):
            zz = (q[hl, L + j] @ k[0].T) / np.sqrt(d)
            np.testing.assert_allclose(p[hl, j, :L + j + 1], np.exp(zz[:L + j + 1] - lse[hl, L + j]), rtol=1e-12)


# --------------------------------------------------------------------------- composition of the steps

def _ref_group_scores(q_l, k_l, L, W, G, mode, softmax):
    """Raw group scores [H_kv, L] of one layer, built outside the oracle: probabilities from torch SDPA
    (identity values) or logits by an explicit dot-product loop, then each head's column sum over the
    window rows, then the reduction over the heads of each group."""
    Hq, d = q_l.shape[0], q_l.shape[-1]
    if softmax:
        c = _sdpa_probs(q_l, k_l, L, W)[:, :, :L].sum(axis=1)            # [Hq, L]
    else:
        c = np.zeros((Hq, L))
        for h in range(Hq):
            for t in range(L):
                c[h, t] = sum(float(np.dot(q_l[h, j], k_l[h // G, t])) for j in range(W)) / math.sqrt(d)
    out = []
    for g in range(k_l.shape[0]):
        heads = c[g * G:(g + 1) * G]
        out.append({"sum": heads.sum(axis=0), "max": heads.max(axis=0),
                    "mean": heads.sum(axis=0) / (G * W)}[mode])
    return np.stack(out)


def _ref_pool(s, k, kind):
    return _pool_loop(s, k) if kind == "max" else _avg_loop(s, k)


def _ref_top(u, k):
    """k best positions by (score desc, index asc), returned ascending."""
    return sorted(sorted(range(len(u)), key=lambda t: (-u[t], t))[:k])


def _ref_pages(u, P):
    n = len(u)
    return np.array([max(u[p * P:min(n, (p + 1) * P)]) for p in range(-(-n // P))])


def _ref_rows(x, idx, P):
    """Rows x[i] (token mode) or the P rows of page i, zero past the end, in list order."""
    out = []
    for i in idx:
        for r in range(i * P, i * P + P):
            out.append(x[r] if r < x.shape[0] else np.zeros(x.shape[1]))
    return np.array(out)


def _workload(**kw):
    import types
    base = dict(group_reduce="sum", pool_k=3, page_size=1, page_reduce="max", k_keep=4, n_recent=0,
                layer_range=None, pool_type="max", score_mode="softmax", head_reduce="group",
                append_window=True)
    base.update(kw)
    return types.SimpleNamespace(**base)


def check_run_sequence_composition(o):
    """run_sequence chains the steps in the order the pages give, on tiny inputs, against outputs rebuilt
    here from SDPA probabilities and loop definitions:

    * token mode: group reduce -> pool -> top k per (layer, KV head) -> window appended -> gather;
    * page mode: group max -> pool -> page max (DELTA key designs 2-3: token scores first, then the page
      score) -> last n_recent prefix pages kept, top k of the others, window pages appended;
    * cross-layer: group sum -> L1 over the prefix per (layer, KV head) -> mean over the inclusive layer
      range -> pool -> one top k per KV head gathered from every layer (LookaheadKV's L1 normalisation;
      CLAA decision 3);
    * all-head: the sum over KV heads of the raw group scores, then the pool, one index per layer
      (CLAA decision 2), here without the window (LookaheadKV's lookahead rows are not kept);
    * pre-softmax logits summed over all heads with average pooling (GemFilter).
    """
    rng = _rng(20)

    def inputs(n_layers, Hq, Hkv, W, L, d, scale=1.6):
        q = _bf16_values(rng.standard_normal((n_layers, Hq, W, d)) * scale)
        k = _bf16_values(rng.standard_normal((n_layers, Hkv, L + W, d)))
        v = _bf16_values(rng.standard_normal((n_layers, Hkv, L + W, d)))
        return q, k, v

    def raw_of(w, q, k, L):
        G = w.h_q // w.h_kv
        return np.stack([_ref_group_scores(q[l], k[l], L, w.window, G, w.group_reduce,
                                           w.score_mode == "softmax") for l in range(w.n_layers)])

    # token mode
    w = _workload(n_layers=2, h_q=4, h_kv=2, window=3, k_keep=5)
    L = 19
    q, k, v = inputs(2, 4, 2, 3, L, 8)
    res = o.run_sequence(w, q, k, v)
    raw = raw_of(w, q, k, L)
    np.testing.assert_allclose(res["raw"], raw, rtol=1e-11, atol=1e-14)
    for l in range(2):
        for g in range(2):
            u = _ref_pool(raw[l, g], 3, "max")
            np.testing.assert_allclose(res["pooled"][l, g], u, rtol=1e-11, atol=1e-14)
            want = _ref_top(u, 5) + list(range(L, L + 3))
            assert list(res["idx"][l, g]) == want, (l, g, list(res["idx"][l, g]), want)
            np.testing.assert_array_equal(res["k_c"][l, g], _ref_rows(k[l, g], want, 1))
            np.testing.assert_array_equal(res["v_c"][l, g], _ref_rows(v[l, g], want, 1))

    # page mode, partial last page shared by prefix and window
    P = 4
    w = _workload(n_layers=2, h_q=4, h_kv=2, window=4, group_reduce="max", page_size=P, k_keep=2, n_recent=1)
    L = 22
    q, k, v = inputs(2, 4, 2, 4, L, 8)
    res = o.run_sequence(w, q, k, v)
    raw = raw_of(w, q, k, L)
    np.testing.assert_allclose(res["raw"], raw, rtol=1e-11, atol=1e-14)
    n_pages = -(-L // P)
    for l in range(2):
        for g in range(2):
            u = _ref_pool(raw[l, g], 3, "max")
            U = _ref_pages(u, P)
            np.testing.assert_allclose(res["pages"][l, g], U, rtol=1e-11, atol=1e-14)
            cand = n_pages - 1
            want = sorted(_ref_top(U[:cand], 2) + [cand]) + list(range(n_pages, -(-(L + 4) // P)))
            assert list(res["idx"][l, g]) == want, (l, g, list(res["idx"][l, g]), want)
            np.testing.assert_array_equal(res["k_c"][l, g], _ref_rows(k[l, g], want, P))

    # cross-layer L1 mean over an inclusive layer range
    w = _workload(n_layers=5, h_q=4, h_kv=2, window=2, k_keep=4, layer_range=(1, 3))
    L = 17
    q, k, v = inputs(5, 4, 2, 2, L, 8)
    res = o.run_sequence(w, q, k, v)
    raw = raw_of(w, q, k, L)
    np.testing.assert_allclose(res["raw"], raw, rtol=1e-11, atol=1e-14)
    for g in range(2):
        S = sum(raw[l, g] / sum(abs(x) for x in raw[l, g]) for l in (1, 2, 3)) / 3.0
        np.testing.assert_allclose(res["combined"][g], S, rtol=1e-11, atol=1e-14)
        u = _ref_pool(S, 3, "max")
        np.testing.assert_allclose(res["pooled"][g], u, rtol=1e-11, atol=1e-14)
        want = _ref_top(u, 4) + [L, L + 1]
        assert list(res["idx"][g]) == want, (g, list(res["idx"][g]), want)
        for l in range(5):
            np.testing.assert_array_equal(res["k_c"][l, g], _ref_rows(k[l, g], want, 1))

    # all-head sum, mean reduce, max pool, window not kept
    w = _workload(n_layers=2, h_q=4, h_kv=2, window=3, group_reduce="mean", head_reduce="all",
                  append_window=False, k_keep=4)
    L = 15
    q, k, v = inputs(2, 4, 2, 3, L, 8)
    res = o.run_sequence(w, q, k, v)
    raw = raw_of(w, q, k, L)
    np.testing.assert_allclose(res["raw"], raw, rtol=1e-11, atol=1e-14)
    for l in range(2):
        u = _ref_pool(raw[l, 0] + raw[l, 1], 3, "max")
        np.testing.assert_allclose(res["pooled"][l], u, rtol=1e-11, atol=1e-14)
        want = _ref_top(u, 4)
        assert list(res["idx"][l]) == want, (l, list(res["idx"][l]), want)
        for g in range(2):
            np.testing.assert_array_equal(res["k_c"][l, g], _ref_rows(k[l, g], want, 1))

    # pre-softmax logits over all heads, average pooling, W = 1
    w = _workload(n_layers=1, h_q=4, h_kv=2, window=1, score_mode="logits", head_reduce="all",
                  pool_type="avg", k_keep=3)
    L = 13
    q, k, v = inputs(1, 4, 2, 1, L, 8)
    res = o.run_sequence(w, q, k, v, with_gather=False)
    raw = raw_of(w, q, k, L)
    np.testing.assert_allclose(res["raw"], raw, rtol=1e-11, atol=1e-13)
    u = _ref_pool(raw[0, 0] + raw[0, 1], 3, "avg")
    np.testing.assert_allclose(res["pooled"][0], u, rtol=1e-11, atol=1e-13)
    assert list(res["idx"][0]) == _ref_top(u, 3) + [L]


ALL_CHECKS = [
    check_probs_match_sdpa,
    check_row_mass_invariant,
    check_identical_keys_closed_form,
    check_hand_worked_example,
    check_one_row_textbook,
    check_planted_key_first,
    check_pool_definition,
    check_page_reduce_definition,
    check_topk_brute_force,
    check_page_selection_rule,
    check_gather,
    check_l1_cross_layer,
    check_block_union,
    check_logits_mode_sdpa_log_ratios,
    check_mean_reduce_and_head_sum,
    check_avg_pool_definition,
    check_layer_max_and_keep_count,
    check_claa_max_buffer,
    check_table_attention_sdpa,
    check_prefill_attention_sdpa,
    check_run_sequence_composition,
]
