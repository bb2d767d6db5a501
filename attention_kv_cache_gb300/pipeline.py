"""The whole selection path for one workload: buffers (torch) plus the C-ABI call sequence.

score -> [combine_layers] -> topk -> compact, and the block-union page table
when the workload has a block mask.  Every step runs in libkvsel's kernels;
this module only allocates device memory and orders the calls on one stream.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import kvsel as K


def desc_for(w, pool_k: Optional[int] = None):
    return K.make_desc(n_layers=w.n_layers, h_q=w.h_q, h_kv=w.h_kv, head_dim=w.head_dim, window=w.window,
                       prefix_lens=w.prefix_lens,
                       group_reduce=K.REDUCE_SUM if w.group_reduce == "sum" else K.REDUCE_MAX,
                       pool_k=w.pool_k if pool_k is None else pool_k, page_size=w.page_size,
                       page_reduce=K.REDUCE_MAX if w.page_reduce == "max" else K.REDUCE_SUM)


def pack(inputs, device="cuda"):
    """Packed device tensors in the library's layouts: q [B, layers, h_q, W, d]; k, v flat (sequences back to back)."""
    q = torch.stack([x for x in inputs.q]).to(device).contiguous()
    if len(inputs.k) == 1:                       # one sequence: a view, no second copy
        return q, inputs.k[0].to(device).reshape(-1), inputs.v[0].to(device).reshape(-1)
    k = torch.cat([x.reshape(-1) for x in inputs.k]).to(device)
    v = torch.cat([x.reshape(-1) for x in inputs.v]).to(device)
    return q, k, v


class Pipeline:
    """Buffers and descriptors of one workload ``w`` (a synth.Workload) on ``device``."""

    def __init__(self, w, device="cuda", n_qblk: Optional[int] = None, n_kvblk_max: Optional[int] = None):
        self.w = w
        self.device = device
        xl = w.layer_range is not None
        self.desc = desc_for(w)
        self.desc_score = desc_for(w, pool_k=1) if xl else self.desc
        ws_bytes = max(K.kvsel_workspace_size(self.desc), K.kvsel_workspace_size(self.desc_score))
        ws = torch.zeros(ws_bytes + K.WS_ALIGN, dtype=torch.uint8, device=device)
        off = (-ws.data_ptr()) % K.WS_ALIGN
        self.ws = ws[off:off + ws_bytes]
        self.ws_bytes = ws_bytes
        P = w.page_size
        n_tok = sum(w.n_layers * w.h_kv * L for L in w.prefix_lens)
        n_pg = sum(w.n_layers * w.h_kv * (-(-L // P)) for L in w.prefix_lens)
        f32 = dict(dtype=torch.float32, device=device)
        self.scores = torch.empty(n_tok, **f32)
        self.page_scores = torch.empty(n_pg, **f32) if P > 1 else None
        self.combined = torch.empty(sum(w.h_kv * L for L in w.prefix_lens), **f32) if xl else None
        self.idx_layers = 1 if xl else w.n_layers
        self.n_sel = w.n_sel()
        self.idx = torch.empty((w.batch, self.idx_layers, w.h_kv, self.n_sel), dtype=torch.int32, device=device)
        rows = self.n_sel * P
        self.k_out = torch.empty((w.batch, w.n_layers, w.h_kv, rows, w.head_dim), dtype=torch.bfloat16,
                                 device=device)
        self.v_out = torch.empty_like(self.k_out)
        self.kv_indptr = self.kv_indices = None
        if w.block_union:
            self.n_qblk = n_qblk or w.q_chunk // w.block
            self.n_kvblk_max = n_kvblk_max or max(-(-L // w.block) for L in w.prefix_lens)
            n_rows = w.batch * w.n_layers * w.h_kv
            self.kv_indptr = torch.empty(n_rows + 1, dtype=torch.int32, device=device)
            self.kv_indices = torch.empty(n_rows * self.n_kvblk_max, dtype=torch.int32, device=device)

    def score(self, q, k, stream=None):
        K.kvsel_score(self.desc_score, q, k, self.scores, self.page_scores, self.ws, self.ws_bytes, stream)

    def select(self, stream=None):
        w = self.w
        if w.layer_range is not None:
            lo, hi = w.layer_range
            K.kvsel_combine_layers(self.desc, self.scores, lo, hi, self.combined, self.ws, self.ws_bytes, stream)
            K.kvsel_topk(self.desc, self.combined, 1, w.k_keep, w.n_recent, self.idx, self.ws, self.ws_bytes, stream)
        else:
            src = self.scores if w.page_size == 1 else self.page_scores
            K.kvsel_topk(self.desc, src, w.n_layers, w.k_keep, w.n_recent, self.idx, self.ws, self.ws_bytes, stream)

    def compact(self, k, v, stream=None):
        K.kvsel_compact(self.desc, k, v, self.idx, self.idx_layers, self.n_sel, self.k_out, self.v_out, self.ws,
                        stream)

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
