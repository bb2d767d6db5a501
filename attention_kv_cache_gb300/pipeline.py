"""The whole selection path for one workload: buffers (torch) plus the C-ABI call sequence.

score -> [aggregate over layers / heads] -> top-k -> compact, and the block-union
page table when the workload has a block mask; the CLAA schedule (per-layer
selections plus a prune index from the token-wise max over a layer buffer) for
workloads that carry one.  Every step runs in libkvsel's kernels; this module
only allocates device memory and orders the calls on one stream.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import kvsel as K

_REDUCE = {"sum": K.REDUCE_SUM, "max": K.REDUCE_MAX, "mean": K.REDUCE_MEAN}


def desc_for(w, pool_k: Optional[int] = None, n_layers: Optional[int] = None, lens_dev=None, len_max: int = 0):
    """Descriptor of workload w: its host prefix lengths, or the device tensor ``lens_dev`` with bound ``len_max``."""
    return K.make_desc(n_layers=w.n_layers if n_layers is None else n_layers, h_q=w.h_q, h_kv=w.h_kv,
                       head_dim=w.head_dim, window=w.window,
                       prefix_lens=None if lens_dev is not None else w.prefix_lens,
                       prefix_lens_dev=lens_dev, prefix_len_max=len_max,
                       group_reduce=_REDUCE[w.group_reduce],
                       pool_k=w.pool_k if pool_k is None else pool_k, page_size=w.page_size,
                       page_reduce=K.REDUCE_MAX if w.page_reduce == "max" else K.REDUCE_SUM,
                       pool_type=K.POOL_AVG if w.pool_type == "avg" else K.POOL_MAX,
                       score_mode=K.SCORE_LOGITS if w.score_mode == "logits" else K.SCORE_SOFTMAX)


def pack(inputs, device="cuda"):
    """Packed device tensors in the library's layouts: q [B, layers, h_q, W, d]; k, v flat (sequences back to back)."""
    q = torch.stack([x for x in inputs.q]).to(device).contiguous()
    if len(inputs.k) == 1:                       # one sequence: a view, no second copy
        return q, inputs.k[0].to(device).reshape(-1), inputs.v[0].to(device).reshape(-1)
    k = torch.cat([x.reshape(-1) for x in inputs.k]).to(device)
    v = torch.cat([x.reshape(-1) for x in inputs.v]).to(device)
    return q, k, v


class Pipeline:
    """Buffers and descriptors of one workload ``w`` (a synth.Workload) on ``device``.

    Per-KV-head selection (``head_reduce == "group"``): scores are pooled by the
    scoring kernel, or combined across a layer range first.  All-head selection
    (``"all"``): raw group scores are summed over every KV head of a layer and
    pooled by kvsel_aggregate, and one selection per layer serves every KV head.
    """

    def __init__(self, w, device="cuda", n_qblk: Optional[int] = None, n_kvblk_max: Optional[int] = None,
                 lens_dev=None, len_max: int = 0):
        """With ``lens_dev`` (int64 device tensor of the prefix lengths) the calls read the lengths on the
        device and every buffer is sized for the bound ``len_max``."""
        if w.claa is not None:
            raise ValueError("CLAA workloads run through ClaaPipeline")
        self.w = w
        self.device = device
        xl = w.layer_range is not None
        self.all_heads = w.head_reduce == "all"
        if self.all_heads and (xl or w.page_size != 1):
            raise ValueError("all-head selection is a token-mode, per-layer path")
        self.desc = desc_for(w, lens_dev=lens_dev, len_max=len_max)
        self.desc_score = (desc_for(w, pool_k=1, lens_dev=lens_dev, len_max=len_max) if (xl or self.all_heads)
                           else self.desc)
        lens = [len_max] * w.batch if lens_dev is not None else list(w.prefix_lens)   # sizes the buffers
        ws_bytes = max(K.kvsel_workspace_size(self.desc), K.kvsel_workspace_size(self.desc_score))
        ws = torch.zeros(ws_bytes + K.WS_ALIGN, dtype=torch.uint8, device=device)
        off = (-ws.data_ptr()) % K.WS_ALIGN
        self.ws = ws[off:off + ws_bytes]
        self.ws_bytes = ws_bytes
        P = w.page_size
        n_tok = sum(w.n_layers * w.h_kv * L for L in lens)
        n_pg = sum(w.n_layers * w.h_kv * (-(-L // P)) for L in lens)
        f32 = dict(dtype=torch.float32, device=device)
        self.scores = torch.empty(n_tok, **f32)
        self.page_scores = torch.empty(n_pg, **f32) if P > 1 else None
        self.combined = torch.empty(sum(w.h_kv * L for L in lens), **f32) if xl else None
        self.agg = torch.empty(sum(w.n_layers * L for L in lens), **f32) if self.all_heads else None
        self.idx_layers = 1 if xl else w.n_layers
        self.idx_heads = 1 if self.all_heads else w.h_kv
        self.n_sel = w.n_sel()
        self.idx = torch.empty((w.batch, self.idx_layers, self.idx_heads, self.n_sel), dtype=torch.int32,
                               device=device)
        rows = self.n_sel * P
        self.k_out = torch.empty((w.batch, w.n_layers, w.h_kv, rows, w.head_dim), dtype=torch.bfloat16,
                                 device=device)
        self.v_out = torch.empty_like(self.k_out)
        self.kv_indptr = self.kv_indices = None
        if w.block_union:
            self.n_qblk = n_qblk or w.q_chunk // w.block
            self.n_kvblk_max = n_kvblk_max or max(-(-L // w.block) for L in lens)
            n_rows = w.batch * w.n_layers * w.h_kv
            self.kv_indptr = torch.empty(n_rows + 1, dtype=torch.int32, device=device)
            self.kv_indices = torch.empty(n_rows * self.n_kvblk_max, dtype=torch.int32, device=device)

    def score(self, q, k, stream=None):
        K.kvsel_score(self.desc_score, q, k, self.scores, self.page_scores, self.ws, self.ws_bytes, stream)

    def select(self, stream=None):
        w = self.w
        app = w.append_window
        if self.all_heads:
            K.kvsel_aggregate(self.desc, self.scores, 0, w.n_layers - 1, K.LAYERS_EACH, K.HEADS_SUM, self.agg,
                              self.ws, self.ws_bytes, stream)
            K.kvsel_select(self.desc, self.agg, w.n_layers, w.k_keep, 0, app, self.idx, self.ws, self.ws_bytes,
                           stream)
        elif w.layer_range is not None:
            lo, hi = w.layer_range
            K.kvsel_combine_layers(self.desc, self.scores, lo, hi, self.combined, self.ws, self.ws_bytes, stream)
            K.kvsel_select(self.desc, self.combined, w.h_kv, w.k_keep, w.n_recent, app, self.idx, self.ws,
                           self.ws_bytes, stream)
        else:
            src = self.scores if w.page_size == 1 else self.page_scores
            K.kvsel_select(self.desc, src, w.n_layers * w.h_kv, w.k_keep, w.n_recent, app, self.idx, self.ws,
                           self.ws_bytes, stream)

    def compact(self, k, v, stream=None):
        if self.idx_heads == self.w.h_kv:
            K.kvsel_compact(self.desc, k, v, self.idx, self.idx_layers, self.n_sel, self.k_out, self.v_out, self.ws,
                            stream)
        else:
            K.kvsel_compact_layers(self.desc, k, v, self.idx, self.idx_layers, 1, 0, self.w.n_layers, self.n_sel,
                                   self.k_out, self.v_out, self.ws, stream)

    def pagetable(self, mask, n_kvblk, stream=None):
        K.kvsel_pagetable(self.desc, mask, self.n_qblk, self.n_kvblk_max, n_kvblk, self.kv_indptr,
                          self.kv_indices, self.ws, self.ws_bytes, stream)

    def run(self, q, k, v, mask=None, n_kvblk=None, stream=None):
        """One pass of the whole path over one batch."""
        self.score(q, k, stream)
        self.select(stream)
        self.compact(k, v, stream)
        if mask is not None:
            self.pagetable(mask, n_kvblk, stream)

    # ---- views of the flat outputs ------------------------------------------------------
    def token_scores(self, b: int) -> torch.Tensor:
        """Pooled (or, with a layer range, raw) scores of sequence b as [n_layers, h_kv, L_b]."""
        w = self.w
        off = sum(w.n_layers * w.h_kv * L for L in w.prefix_lens[:b])
        L = w.prefix_lens[b]
        return self.scores[off:off + w.n_layers * w.h_kv * L].view(w.n_layers, w.h_kv, L)

    def page_view(self, b: int) -> torch.Tensor:
        w = self.w
        P = w.page_size
        off = sum(w.n_layers * w.h_kv * (-(-L // P)) for L in w.prefix_lens[:b])
        n = -(-w.prefix_lens[b] // P)
        return self.page_scores[off:off + w.n_layers * w.h_kv * n].view(w.n_layers, w.h_kv, n)

    def combined_view(self, b: int) -> torch.Tensor:
        w = self.w
        off = sum(w.h_kv * L for L in w.prefix_lens[:b])
        L = w.prefix_lens[b]
        return self.combined[off:off + w.h_kv * L].view(w.h_kv, L)


class ClaaPipeline:
    """CLAA selection of one prompt (CLAA, 'Three design decisions' and 'Complete flow and cost'),
    run by kvsel_claa_select: layers m .. l_p are scored with the observation window, each keeps
    its own top-k (k from the keep rate) and its cache is compacted; at l_p the token-wise max over
    the buffered layers picks the sequence prune index.  The schedule's sizes (scored layers, the
    buffer, k) come from kvsel_claa_shape; this class only allocates the buffers.
    """

    def __init__(self, w, device="cuda"):
        if w.claa is None or w.batch != 1:
            raise ValueError("a CLAA workload of one prompt")
        self.w = w
        self.device = device
        m, lp, nbuf, rate = w.claa
        self.params = K.ClaaParams(m, lp, nbuf, rate)
        self.desc = desc_for(w)
        shape = K.kvsel_claa_shape(self.desc, self.params)
        self.m, self.lp = m, lp
        self.n_sc = shape.n_scored                          # layers scored and compacted
        self.buf_lo = shape.buffer_lo - m                   # buffer, relative to layer m
        self.k = shape.k
        self.n_sel = shape.n_sel
        L = w.prefix_lens[0]
        ws = torch.zeros(shape.ws_bytes + K.WS_ALIGN, dtype=torch.uint8, device=device)
        off = (-ws.data_ptr()) % K.WS_ALIGN
        self.ws = ws[off:off + shape.ws_bytes]
        self.ws_bytes = shape.ws_bytes
        f32 = dict(dtype=torch.float32, device=device)
        self.scores = torch.empty((self.n_sc, w.h_kv, L), **f32)       # raw group scores
        self.layer_scores = torch.empty((self.n_sc, L), **f32)          # pooled all-head score per layer
        self.prune_scores = torch.empty((1, L), **f32)                  # pooled max over the buffer
        self.idx = torch.empty((1, self.n_sc, 1, self.n_sel), dtype=torch.int32, device=device)
        self.prune_idx = torch.empty((1, 1, self.n_sel), dtype=torch.int32, device=device)
        self.k_out = torch.empty((1, self.n_sc, w.h_kv, self.n_sel, w.head_dim), dtype=torch.bfloat16, device=device)
        self.v_out = torch.empty_like(self.k_out)

    def run(self, q, k, v, stream=None):
        """q [1, n_layers, h_q, W, d]; k, v the prompt's caches (flat, layout of the library)."""
        K.kvsel_claa_select(self.desc, self.params, q, k, v, self.scores, self.layer_scores, self.prune_scores,
                            self.idx, self.prune_idx, self.k_out, self.v_out, self.ws, self.ws_bytes, stream)
