"""fp64 CPU oracle for window-attention KV selection.

TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this module; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use it.  It shares no code with the CUDA path and imports nothing from it.

Each function writes out the plain definition of one step, in float64, with
numpy (a matrix product and a sort are the only library primitives used).
Inputs arrive as bf16 values (from the workload generator) and are decoded to
float64 exactly.

Sources (page title, then the section / equation the step follows):

* ClusterAttn: KV Cache Compression under Intrinsic Attention Clustering (ACL
  2025), 'Background and key observations' (背景知识与关键观察): the feature
  aggregation equations W_win = Q[:, -L_win:] K^T, the window mask M_win, the
  softmax A^m_win and the column sum P = sum over the window rows of
  A^m_win[:, i, :L_pre]; 'Method details' (方法细节): the compressed prefix is
  concatenated with the full observation window.
* CLAA: cross-layer attention aggregation (2026), 'Three representative
  token-ranking methods' (FastKV) and 'Three design decisions', decision 2:
  post-softmax window probabilities summed over the window queries and heads;
  decision 3 (Eq. 6): per-token aggregation across layers; 'Oracle
  construction': 1-D pooling with kernel 7 after the aggregation.
* DELTA: Dynamic Layer-Aware Token Attention (ACL 2026 Findings), 'Key
  designs' 2 and 3: token score = max over heads, page score over the P = 16
  tokens of a page, last L pages kept plus the top K - L of the remaining pages.
* LookaheadKV (2026), 'Background: KL divergence and ListNet': L1
  normalisation s / ||s||_1 of importance scores.
* CompactAttention: Accelerating Chunked Prefill with Block-Union KV Selection,
  'Core method' and 'Method steps' (2): Q-block union, intra-group union and
  the per-group table T_{b,g} = { j | G_{b,g,j} = 1 }.
* CLAA, 'Three representative token-ranking methods' (GemFilter): the
  pre-softmax attention of the last prompt token, summed over all heads;
  'Three design decisions' (m = 4 deferred layers, per-layer window scores in
  a rolling buffer of n = 4, token-wise max at the pruning layer l_p = 15) and
  'Complete flow and cost' (per-layer top-k by keep rate and gather of the
  cache; a sequence prune index at l_p); 'Experimental setup': average pooling
  with kernel 7 for every method.
* LookaheadKV, 'Method steps': the lookahead rows' attention to the prompt is
  averaged, pooled, and the top K kept.
* CLAA, 'Complete flow and cost' (engineering detail 1): the keys that score the
  window are the prefill's own intermediate results; the prefill attention is
  causal softmax attention over the prompt, o_i = sum_{t <= i} softmax_t(q_i k_t /
  sqrt(d)) v_t, and its per-row log-sum-exp is what the window scores need.
* CompactAttention, 'Method steps' (3): the selected KV blocks are read in
  place by a paged dense-attention kernel through kv_indptr / kv_indices;
  DELTA, 'Overall framework': sparse layers attend only over the selected page
  set.  The attention itself is softmax(q K^T / sqrt(d)) V over those rows.

Readings taken where the pages are silent or garbled (each is also listed in
the design notes):

* The window mask is additive-causal: window row j (absolute position L + j)
  sees every prefix key and window keys 0..j; the softmax runs over that full
  row; only prefix columns t < L are emitted.
* Scale is 1/sqrt(d) (the standard attention scale the CLAA page names).
* Query head h belongs to KV head g = h // (H_q / H_kv).
* Max-over-heads with W > 1 is max_h (sum_j p): the column mass of each head
  first, then the max over the heads of the group.
* Pooling is max-pooling, centred, stride 1, same length, out-of-range
  neighbours ignored, over prefix columns only.
* A page's score reduces the pooled token scores of its tokens (max by
  default, sum as the DELTA page prints it); the last page may be partial.
* Ranking is by (score descending, index ascending).
* Selected entries are returned in ascending original position, then the
  observation window (token mode) or its pages (page mode) is appended.
* Cross-layer: each layer's group score is L1-normalised over t < L, then the
  mean over an inclusive layer range is taken, then pooled.
* Average pooling divides by the number of in-range neighbours (out-of-range
  neighbours are ignored, as for the max).
* Pre-softmax scores sum the scaled logits of the window rows (W = 1 is
  GemFilter's last token); the keys stay those of the prefix.
* 'mean' group reduce = the group sum divided by G * W (the mean over the
  group's window rows and heads).
* A keep rate r maps to k = floor(r * L + 1/2) prefix tokens (round half up),
  clipped to [0, L]; the observation window is appended as in token mode.
* Attention over a page / block table: a query row attends to every row of
  every listed block (block b covers rows bP .. bP + P - 1, rows past the
  cache's end do not exist), with no causal mask (decode-style queries come
  after every selected key).
* CLAA over an offline prompt: layers m .. l_p are scored with the window
  (sum over window rows and all heads, softmax), each layer's pooled scores give
  its own top-k, and the token-wise max over the last n buffered layers (up to
  and including l_p, not before m), pooled, gives the sequence prune index.
  Layers after l_p run on the pruned sequence, which only a model forward
  produces; they are scored like any other layer on their own inputs.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    """bf16 / fp32 torch tensor or array -> float64 ndarray (exact)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        return x.double().numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------- scoring

def window_logits(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """z[r, t] = <q_r, k_t> / sqrt(d) for every window query row r and key t.

    ClusterAttn 'Background and key observations', W_win = Q[:, -L_win:] K^T,
    with the 1/sqrt(d_k) scale of standard attention.
    q: [R, d] float64, k: [N, d] float64 -> [R, N].
    """
    d = q.shape[-1]
    return (q @ k.T) / np.sqrt(d)


def window_mask(L: int, W: int) -> np.ndarray:
    """visible[j, t] for window row j and key t < L + W: all prefix keys, window keys 0..j."""
    t = np.arange(L + W)[None, :]
    j = np.arange(W)[:, None]
    return t <= L + j


def window_probs(q_group: np.ndarray, k_head: np.ndarray, L: int) -> np.ndarray:
    """A^m_win: masked softmax rows of one GQA group.

    q_group: [G, W, d] window queries of the G query heads that share KV head
    k_head: [L + W, d].  Returns p [G, W, L + W]; each row sums to one over
    its visible keys and is zero on masked ones.
    """
    G, W, d = q_group.shape
    z = window_logits(q_group.reshape(G * W, d), k_head).reshape(G, W, L + W)
    vis = window_mask(L, W)[None, :, :]
    z = np.where(vis, z, -np.inf)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def column_mass(p: np.ndarray, L: int) -> np.ndarray:
    """P: column sum over the window rows, restricted to prefix columns :L.  [G, W, N] -> [G, L]."""
    return p[:, :, :L].sum(axis=1)


def logit_mass(q_group: np.ndarray, k_head: np.ndarray, L: int) -> np.ndarray:
    """Pre-softmax column sum c[h, t] = sum_j z[h, j, t] over prefix keys t < L.

    CLAA 'Three representative token-ranking methods' (GemFilter): the raw
    attention logit of the last prompt token (W = 1) for every prompt key.
    q_group: [G, W, d], k_head: [L + W, d] -> [G, L].  Prefix keys are visible
    to every window row, so no mask applies.
    """
    G, W, d = q_group.shape
    z = window_logits(q_group.reshape(G * W, d), k_head[:L]).reshape(G, W, L)
    return z.sum(axis=1)


def group_reduce(c: np.ndarray, mode: str, W: int = 1) -> np.ndarray:
    """Reduce the per-head column mass [G, L] over the heads of one group: 'sum', 'max' or 'mean'
    (the sum divided by G * W, the mean over the group's W window rows and G heads)."""
    if mode == "sum":
        return c.sum(axis=0)
    if mode == "max":
        return c.max(axis=0)
    if mode == "mean":
        return c.sum(axis=0) / (c.shape[0] * W)
    raise ValueError(mode)


def group_scores(q_group, k_head, L: int, mode: str, softmax: bool = True) -> np.ndarray:
    """s[t], t < L, for one (layer, KV head): probabilities (or raw logits) -> column mass -> group reduce."""
    c = column_mass(window_probs(q_group, k_head, L), L) if softmax else logit_mass(q_group, k_head, L)
    return group_reduce(c, mode, q_group.shape[1])


def max_pool(s: np.ndarray, k: int) -> np.ndarray:
    """u[t] = max of s over [t - r, t + r] intersected with [0, len), r = (k - 1) / 2 (last axis)."""
    if k % 2 != 1 or k < 1:
        raise ValueError("pool width must be odd")
    r = (k - 1) // 2
    n = s.shape[-1]
    out = s.copy()
    for off in range(1, r + 1):
        if off >= n:
            break
        out[..., :-off] = np.maximum(out[..., :-off], s[..., off:])
        out[..., off:] = np.maximum(out[..., off:], s[..., :-off])
    return out


def avg_pool(s: np.ndarray, k: int) -> np.ndarray:
    """u[t] = mean of s over [t - r, t + r] intersected with [0, len), r = (k - 1) / 2 (last axis).

    CLAA 'Oracle construction' and 'Experimental setup': 1-D average pooling,
    kernel 7.  Only in-range neighbours are counted.
    """
    if k % 2 != 1 or k < 1:
        raise ValueError("pool width must be odd")
    r = (k - 1) // 2
    n = s.shape[-1]
    tot = s.copy()
    cnt = np.ones(n)
    for off in range(1, r + 1):
        if off >= n:
            break
        tot[..., :-off] += s[..., off:]
        tot[..., off:] += s[..., :-off]
        cnt[:-off] += 1
        cnt[off:] += 1
    return tot / cnt


def pool(s: np.ndarray, k: int, kind: str = "max") -> np.ndarray:
    """Max or average pooling of width k along the last axis."""
    if kind == "max":
        return max_pool(s, k)
    if kind == "avg":
        return avg_pool(s, k)
    raise ValueError(kind)


def page_reduce(u: np.ndarray, P: int, mode: str = "max") -> np.ndarray:
    """U[p] over the tokens [pP, min((p+1)P, L)) of each page (last axis; last page may be partial)."""
    n = u.shape[-1]
    n_pages = -(-n // P)
    pad = n_pages * P - n
    fill = -np.inf if mode == "max" else 0.0
    x = np.concatenate([u, np.full(u.shape[:-1] + (pad,), fill)], axis=-1)
    x = x.reshape(u.shape[:-1] + (n_pages, P))
    if mode == "max":
        return x.max(axis=-1)
    if mode == "sum":
        return x.sum(axis=-1)
    raise ValueError(mode)


def l1_normalise(s: np.ndarray) -> np.ndarray:
    """s / ||s||_1 along the last axis (LookaheadKV's normalisation of importance scores)."""
    return s / np.abs(s).sum(axis=-1, keepdims=True)


def cross_layer_mean(s_layers: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Mean over layers lo..hi (inclusive) of the L1-normalised scores.  s_layers: [n_layers, ..., L]."""
    return l1_normalise(s_layers[lo:hi + 1]).mean(axis=0)


def head_sum(s: np.ndarray) -> np.ndarray:
    """Sum over every KV head of a layer's group scores [..., H_kv, L] -> [..., L]: the sum over
    all attention heads that FastKV, CLAA and GemFilter score with (CLAA, decision 2)."""
    return s.sum(axis=-2)


def layer_max(s_layers: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Token-wise max over layers lo..hi (inclusive) of s_layers [n_layers, ..., L] (CLAA Eq. 6)."""
    return s_layers[lo:hi + 1].max(axis=0)


def keep_count(keep_rate: float, L: int) -> int:
    """Prefix tokens kept for a keep rate: floor(r * L + 1/2), clipped to [0, L]."""
    return int(min(L, max(0, np.floor(keep_rate * L + 0.5))))


# --------------------------------------------------------------------------- selection

def rank(scores: np.ndarray) -> np.ndarray:
    """Positions ordered by (score descending, index ascending), by a full stable sort."""
    n = scores.shape[-1]
    return np.lexsort((np.arange(n), -scores))


def select_tokens(u: np.ndarray, k: int, L: int, W: int) -> np.ndarray:
    """Top-k prefix tokens of one row, ascending, followed by the window positions L..L+W-1."""
    top = np.sort(rank(u[:L])[:k])
    return np.concatenate([top, np.arange(L, L + W)]).astype(np.int64)


def select_pages(U: np.ndarray, k: int, n_recent: int, L: int, W: int, P: int) -> np.ndarray:
    """DELTA page rule for one row, then the window's pages.

    The last ``n_recent`` prefix pages are always kept; the top k of the
    remaining prefix pages are added; the result is sorted ascending and the
    pages holding window tokens beyond the prefix pages are appended.
    """
    n_pages = -(-L // P)
    cand = n_pages - n_recent
    top = rank(U[:cand])[:k]
    keep = np.sort(np.concatenate([top, np.arange(cand, n_pages)]))
    wpages = np.arange(n_pages, -(-(L + W) // P))
    return np.concatenate([keep, wpages]).astype(np.int64)


def gather_rows(x: np.ndarray, idx: np.ndarray, page_size: int = 1) -> np.ndarray:
    """Rows of x [N, d] at idx (token mode) or the P rows of each page (page mode); rows past N are 0."""
    if page_size == 1:
        return x[idx]
    rows = (idx[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)
    out = np.zeros((rows.size,) + x.shape[1:], dtype=x.dtype)
    ok = rows < x.shape[0]
    out[ok] = x[rows[ok]]
    return out


# --------------------------------------------------------------------------- attention over a table

def table_rows(blocks: np.ndarray, P: int, n_rows: int) -> np.ndarray:
    """Cache rows named by a block list: rows bP .. bP + P - 1 of each block b, in list order, < n_rows."""
    rows = (np.asarray(blocks, np.int64)[:, None] * P + np.arange(P)[None, :]).reshape(-1)
    return rows[rows < n_rows]


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """o[r] = softmax_t(<q_r, k_t> / sqrt(d)) v_t over the given cache rows t.  q [R, d] -> [R, d]."""
    z = window_logits(q, k[rows])
    z = z - z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ v[rows]


def prefill_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """Causal attention of every prompt row.  q [H_q, N, d], k / v [H_kv, N, d] (GQA map h -> h // G).

    Returns o [H_q, N, d] and lse [H_q, N], the natural-log log-sum-exp of each row's scaled logits
    over its visible keys t <= i.
    """
    Hq, N, d = q.shape
    G = Hq // k.shape[0]
    vis = np.arange(N)[None, :] <= np.arange(N)[:, None]
    o = np.zeros_like(q)
    lse = np.zeros((Hq, N))
    for h in range(Hq):
        z = np.where(vis, window_logits(q[h], k[h // G]), -np.inf)
        m = z.max(axis=-1, keepdims=True)
        e = np.exp(z - m)
        ssum = e.sum(axis=-1, keepdims=True)
        o[h] = (e / ssum) @ v[h // G]
        lse[h] = (m + np.log(ssum))[:, 0]
    return o, lse


def prefill_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows):
    """prefill_attention restricted to the listed rows, for prompts whose full N x N logits do not fit:
    o [H_q, len(rows), d] and lse [H_q, len(rows)], row i attending to keys t <= i.  q [H_q, N, d],
    k / v [H_kv, N, d] (any dtype)."""
    Hq, d = q.shape[0], q.shape[-1]
    G = Hq // k.shape[0]
    rows = [int(i) for i in rows]
    o = np.zeros((Hq, len(rows), d))
    lse = np.zeros((Hq, len(rows)))
    for h in range(Hq):
        kh, vh = _f64(k[h // G]), _f64(v[h // G])
        qh = _f64(q[h])
        for n, i in enumerate(rows):
            z = window_logits(qh[i:i + 1], kh[:i + 1])[0]
            m = z.max()
            e = np.exp(z - m)
            ssum = e.sum()
            o[h, n] = (e / ssum) @ vh[:i + 1]
            lse[h, n] = m + np.log(ssum)
    return o, lse


# --------------------------------------------------------------------------- block union

def block_union(mask: np.ndarray, h_kv: int, n_kv: int):
    """Per-group KV block list of one (sequence, layer).

    mask: [H_q, n_qblk, >= n_kv] of 0/1.  Q-block union Mbar[h, j] = OR_i M[h, i, j];
    intra-group union G[g, j] = OR over h in group g of Mbar[h, j]; T_g = { j : G[g, j] = 1 }.
    Returns a list of h_kv ascending int arrays.
    """
    H = mask.shape[0]
    Gsz = H // h_kv
    out = []
    for g in range(h_kv):
        hit = np.zeros(n_kv, dtype=bool)
        for h in range(g * Gsz, (g + 1) * Gsz):
            for i in range(mask.shape[1]):
                hit |= mask[h, i, :n_kv] != 0
        out.append(np.nonzero(hit)[0].astype(np.int64))
    return out


def block_union_csr(mask: np.ndarray, h_kv: int, n_kv: list):
    """CSR over rows (b, layer, g): kv_indptr [B*layers*h_kv + 1], kv_indices.  mask: [B, layers, H_q, n_qblk, nmax]."""
    lists = []
    for b in range(mask.shape[0]):
        for layer in range(mask.shape[1]):
            lists.extend(block_union(mask[b, layer], h_kv, n_kv[b]))
    indptr = np.zeros(len(lists) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum([len(x) for x in lists])
    indices = np.concatenate(lists) if lists else np.zeros(0, dtype=np.int64)
    return indptr, indices


# --------------------------------------------------------------------------- whole workload

def score_unit(q_layer, k_layer, g: int, G: int, L: int, mode: str, softmax: bool = True) -> np.ndarray:
    """Raw group scores of (layer, KV head g): q_layer [H_q, W, d], k_layer [H_kv, L+W, d] (any dtype)."""
    qg = _f64(q_layer[g * G:(g + 1) * G])
    kh = _f64(k_layer[g])
    return group_scores(qg, kh, L, mode, softmax)


def claa_sequence(q, k, L: int, W: int, G: int, h_kv: int, defer: int, prune_layer: int, agg_window: int,
                  keep_rate: float, pool_k: int = 7, pool_kind: str = "avg"):
    """CLAA selection for one prompt, following 'Three design decisions' and 'Complete flow and cost'.

    q [n_layers, H_q, W, d], k [n_layers, H_kv, L + W, d].  For every layer l in
    defer .. prune_layer: the window score of each prefix token (softmax
    probabilities summed over the window rows and all heads), its pooled form,
    and the layer's own top-k (k from the keep rate) followed by the window.
    At prune_layer: the token-wise max over the buffered layers
    max(defer, prune_layer - agg_window + 1) .. prune_layer, pooled, and its
    top-k followed by the window: the sequence prune index.
    """
    kc = keep_count(keep_rate, L)
    layer_s, layer_idx = {}, {}
    for l in range(defer, prune_layer + 1):
        s = head_sum(np.stack([score_unit(q[l], k[l], g, G, L, "sum") for g in range(h_kv)]))
        layer_s[l] = s
        layer_idx[l] = select_tokens(pool(s, pool_k, pool_kind), kc, L, W)
    lo = max(defer, prune_layer - agg_window + 1)
    buf = np.stack([layer_s[l] for l in range(lo, prune_layer + 1)])
    agg = layer_max(buf, 0, buf.shape[0] - 1)
    u = pool(agg, pool_k, pool_kind)
    return {"layer_scores": layer_s, "layer_idx": layer_idx, "agg": agg, "prune_scores": u,
            "prune_idx": select_tokens(u, kc, L, W), "k": kc, "buffer": (lo, prune_layer)}


def run_sequence(w, q, k, v=None, with_gather: bool = True, layers=None):
    """Every output of the path for one sequence of workload ``w`` (an object with the
    Workload fields).  q [n_layers, H_q, W, d], k/v [n_layers, H_kv, L+W, d].

    Returns a dict: 'raw' [n_layers, H_kv, L] group scores, 'pooled' (per layer
    or, with a layer range, [H_kv, L] after the cross-layer mean; with all-head
    selection [n_layers, L] after the sum over KV heads), 'pages' [.., n_pages]
    in page mode, 'idx' selected positions (or pages), and, with
    ``with_gather``, 'k_c' / 'v_c' compacted rows.
    """
    L = int(k.shape[2]) - w.window
    W, G, Hkv = w.window, w.h_q // w.h_kv, w.h_kv
    Wapp = W if getattr(w, "append_window", True) else 0
    softmax = getattr(w, "score_mode", "softmax") == "softmax"
    kind = getattr(w, "pool_type", "max")
    all_heads = getattr(w, "head_reduce", "group") == "all"
    layers = range(w.n_layers) if layers is None else layers
    raw = np.stack([np.stack([score_unit(q[l], k[l], g, G, L, w.group_reduce, softmax) for g in range(Hkv)])
                    for l in layers])
    out = {"raw": raw}
    if all_heads:
        u = pool(head_sum(raw), w.pool_k, kind)                  # [layers, L]
        out["pooled"] = u
        out["idx"] = np.stack([select_tokens(u[i], w.k_keep, L, Wapp) for i in range(u.shape[0])])
    elif w.layer_range is not None:
        lo, hi = w.layer_range
        s = cross_layer_mean(raw, lo, hi)                       # [H_kv, L]
        u = pool(s, w.pool_k, kind)
        idx = np.stack([select_tokens(u[g], w.k_keep, L, Wapp) for g in range(Hkv)])
        out.update(combined=s, pooled=u, idx=idx)
    else:
        u = pool(raw, w.pool_k, kind)                            # [layers, H_kv, L]
        out["pooled"] = u
        if w.page_size == 1:
            idx = np.stack([np.stack([select_tokens(u[i, g], w.k_keep, L, Wapp) for g in range(Hkv)])
                            for i in range(u.shape[0])])
        else:
            U = page_reduce(u, w.page_size, w.page_reduce)
            out["pages"] = U
            idx = np.stack([np.stack([select_pages(U[i, g], w.k_keep, w.n_recent, L, Wapp, w.page_size)
                                      for g in range(Hkv)]) for i in range(u.shape[0])])
        out["idx"] = idx
    if with_gather and v is not None:
        P = w.page_size
        kc, vc = [], []
        for i, l in enumerate(layers):
            kl, vl = [], []
            for g in range(Hkv):
                if all_heads:
                    ii = out["idx"][i]
                elif w.layer_range is not None:
                    ii = out["idx"][g]
                else:
                    ii = out["idx"][i, g]
                kl.append(gather_rows(_f64(k[l, g]), ii, P))
                vl.append(gather_rows(_f64(v[l, g]), ii, P))
            kc.append(np.stack(kl)); vc.append(np.stack(vl))
        out["k_c"] = np.stack(kc)
        out["v_c"] = np.stack(vc)
    return out
