"""Seeded synthetic workloads for window-attention KV selection.

This module is the one place that makes inputs. Both the CUDA path (through
the Python binding) and the fp64 oracle consume what it returns; it holds none
of the method's arithmetic (no logits, softmax, pooling or selection), only
random numbers and the structure the pages' workloads have:

* Q/K/V drawn i.i.d. N(0, 1) in fp32 and rounded to bf16, shaped like the
  models the pages run (LLaMA-3.1-8B: 32 layers, 32 query / 8 KV heads,
  d = 128; a 70B-shaped model: 80 layers, 64 / 8 heads).
* "Intrinsic attention clusters" (ClusterAttn, 'Background and key
  observations': high-scoring tokens gather in contiguous runs) are planted as
  runs of 64 consecutive prefix keys of one (layer, KV head) shifted by
  1.5 * sqrt(d) along the unit mean direction of that group's window queries,
  in fp32 before the bf16 rounding.
* For the ragged batch: prefix lengths uniform in [8192, 32768], and a binary
  block mask M[b, layer, h, i, j] (CompactAttention, 'Method steps', step 1: a
  selector's 2-D block mask) with about 10 % ones laid out in runs of 2..8
  consecutive KV blocks, each run shared by all Q blocks of the head with
  probability 1/2 and redrawn per Q block otherwise.

Everything is drawn from ``torch.Generator`` streams seeded per workload, on
the device the caller names; callers that need the same data on two devices
generate once and copy.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

SEED_BASE = 0x6B7673656C


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and selection parameters of one synthetic workload.

    ``prefix_lens`` holds L_b for each sequence b (the prompt has L_b prefix
    tokens followed by ``window`` observation-window tokens).  ``k_keep`` is a
    token count in token mode (``page_size == 1``) and a page count in page
    mode.  ``layer_range`` = (lo, hi), inclusive, turns on the cross-layer
    L1-normalised mean before one shared top-k.
    """

    name: str
    index: int
    n_layers: int
    h_q: int
    h_kv: int
    head_dim: int
    window: int
    prefix_lens: tuple
    group_reduce: str = "sum"          # "sum" | "max" | "mean" over the query heads of a group
    pool_k: int = 7                    # odd pool width, 1 = off
    page_size: int = 1                 # 1 = token mode, P > 1 = page mode
    page_reduce: str = "max"           # "max" | "sum" over the tokens of a page
    k_keep: int = 64
    n_recent: int = 0                  # recency pages kept in page mode
    n_clusters: int = 0                # planted 64-token clusters per (layer, KV head)
    cluster_len: int = 64
    layer_range: Optional[tuple] = None
    # block-union page table (ragged batch)
    block_union: bool = False
    q_chunk: int = 1024
    block: int = 64
    mask_density: float = 0.10
    # scoring variants
    pool_type: str = "max"             # "max" | "avg" pooling
    score_mode: str = "softmax"        # "softmax" | "logits" (pre-softmax, GemFilter)
    head_reduce: str = "group"         # "group": one selection per KV head; "all": sum over every KV head
    append_window: bool = True         # False: the window rows are not kept (LookaheadKV's lookahead rows)
    # CLAA schedule: (defer m, pruning layer l_p, buffer n, keep rate); k_keep then comes from the rate
    claa: Optional[tuple] = None

    @property
    def batch(self) -> int:
        return len(self.prefix_lens)

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    def n_keys(self, b: int) -> int:
        return self.prefix_lens[b] + self.window

    def n_sel(self) -> int:
        """Selected entries per (sequence, layer, KV head) row of the index output."""
        win = self.window if self.append_window else 0
        if self.page_size == 1:
            return self.k_keep + win
        return self.k_keep + self.n_recent + win // self.page_size

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _ragged_lens(n: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator().manual_seed(seed ^ 0x5EED)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


# The five workloads.  Indices follow the order they are listed in.
TINY = Workload("tiny_1l_h4x2_d64_L512_W16", 0, 1, 4, 2, 64, 16, (512,),
                group_reduce="sum", pool_k=7, k_keep=64)
LLAMA8B_32K = Workload("llama8b_32l_h32x8_d128_L32768_W32", 1, 32, 32, 8, 128, 32, (32768,),
                       group_reduce="sum", pool_k=7, k_keep=1024, n_clusters=8)
LLAMA8B_128K_PAGED = Workload("llama8b_32l_h32x8_d128_L131072_W32_paged16", 2, 32, 32, 8, 128, 32,
                              (131072,), group_reduce="max", pool_k=7, page_size=16,
                              page_reduce="max", k_keep=128, n_recent=4, n_clusters=32)
RAGGED_B8 = Workload("ragged_b8_32l_h32x8_d128_L8k-32k_W32", 3, 32, 32, 8, 128, 32,
                     _ragged_lens(8, 8192, 32768, SEED_BASE + 3),
                     group_reduce="sum", pool_k=7, k_keep=1024, n_clusters=8, block_union=True)
LLAMA70B_64K_XLAYER = Workload("llama70b_80l_h64x8_d128_L65536_W32_xlayer", 4, 80, 64, 8, 128, 32,
                               (65536,), group_reduce="sum", pool_k=7, k_keep=4096, n_clusters=8,
                               layer_range=(8, 79))

WORKLOADS = (TINY, LLAMA8B_32K, LLAMA8B_128K_PAGED, RAGGED_B8, LLAMA70B_64K_XLAYER)

# Scoring variants of the pages on the LLaMA-8B 32K shape.
# CLAA: W = 8 window, softmax mass summed over the window and all heads, average pool 7, m = 4
# deferred layers, a buffer of n = 4 layers, pruning layer l_p = 15, keep rate 0.2 ('Three design
# decisions'; 'Experimental setup').
CLAA_LLAMA8B_32K = Workload("claa_llama8b_32l_h32x8_d128_L32768_W8_keep0.2", 5, 32, 32, 8, 128, 8, (32768,),
                            group_reduce="sum", pool_k=7, pool_type="avg", head_reduce="all", n_clusters=8,
                            claa=(4, 15, 4, 0.2))
# GemFilter: the last prompt token's pre-softmax logits summed over all heads, average pool 7, 1024 kept.
GEMFILTER_LLAMA8B_32K = Workload("gemfilter_llama8b_32l_h32x8_d128_L32768_W1", 6, 32, 32, 8, 128, 1, (32768,),
                                 group_reduce="sum", pool_k=7, pool_type="avg", score_mode="logits",
                                 head_reduce="all", k_keep=1024, n_clusters=8)
# LookaheadKV: 32 lookahead rows averaged per KV head, pooled, top 128 per head; the lookahead rows
# themselves are not kept.
LOOKAHEAD_LLAMA8B_32K = Workload("lookahead_llama8b_32l_h32x8_d128_L32768_W32_C128", 7, 32, 32, 8, 128, 32,
                                 (32768,), group_reduce="mean", pool_k=7, pool_type="avg", k_keep=128,
                                 append_window=False, n_clusters=8)

# The group max over heads of 24 window rows (a window that is not a power of two): the shape the
# tensor-core scoring does not cover, served by the CUDA-core kernels.
MAXW24_LLAMA8B_32K = Workload("maxw24_llama8b_32l_h32x8_d128_L32768_W24", 8, 32, 32, 8, 128, 24, (32768,),
                              group_reduce="max", pool_k=7, k_keep=1024, n_clusters=8)

VARIANTS = (CLAA_LLAMA8B_32K, GEMFILTER_LLAMA8B_32K, LOOKAHEAD_LLAMA8B_32K, MAXW24_LLAMA8B_32K)


def by_name(name: str) -> Workload:
    for w in WORKLOADS + VARIANTS:
        if w.name == name:
            return w
    raise KeyError(name)


# --------------------------------------------------------------------------- tensors

@dataclasses.dataclass
class Inputs:
    """Q, K, V of a workload.

    Uniform batch (one sequence): q [n_layers, h_q, W, d], k / v
    [n_layers, h_kv, L + W, d].  Ragged batch: lists with one such tensor per
    sequence (the binding packs them).  ``mask`` is [B, n_layers, h_q, n_qblk,
    n_kvblk_max] uint8 or None; ``n_kvblk`` the per-sequence KV-block counts.
    """

    w: Workload
    q: list
    k: list
    v: list
    clusters: list            # per sequence: LongTensor [n_layers, h_kv, n_clusters] of run starts
    mask: Optional[torch.Tensor] = None
    n_kvblk: Optional[list] = None


def _cluster_starts(w: Workload, L: int, gen: torch.Generator, device) -> torch.Tensor:
    """Non-overlapping run starts: one run inside each of n_clusters equal slots of [0, L).  [1, h_kv, n]."""
    n = w.n_clusters
    slot = L // n
    if slot < w.cluster_len:
        raise ValueError("prefix too short for the planted clusters")
    off = torch.randint(0, slot - w.cluster_len + 1, (1, w.h_kv, n), generator=gen, device=device)
    base = torch.arange(n, device=device) * slot
    return base + off


def _layer_generator(w: Workload, b: int, layer: int, device) -> torch.Generator:
    """Each (sequence, layer) draws from its own stream, so any layer can be regenerated alone."""
    return torch.Generator(device=device).manual_seed(w.seed * 1_000_003 + b * 10_007 + layer + 1)


def make_queries(w: Workload, b: int, device="cpu") -> torch.Tensor:
    """Window queries of sequence b: [n_layers, h_q, W, d] bf16."""
    gen = torch.Generator(device=device).manual_seed(w.seed * 1_000_003 + b * 10_007)
    q32 = torch.randn((w.n_layers, w.h_q, w.window, w.head_dim), generator=gen, device=device,
                      dtype=torch.float32)
    return q32.to(torch.bfloat16)


def make_layer(w: Workload, b: int, layer: int, q: torch.Tensor, device="cpu"):
    """K, V ([h_kv, L_b + W, d] bf16) and the planted run starts ([h_kv, n_clusters]) of one layer.

    ``q`` is the sequence's query tensor from make_queries (the cluster
    direction is the mean of each group's window queries of this layer).
    """
    L, W, d = w.prefix_lens[b], w.window, w.head_dim
    n = L + W
    gen = _layer_generator(w, b, layer, device)
    k32 = torch.randn((w.h_kv, n, d), generator=gen, device=device, dtype=torch.float32)
    starts = torch.zeros((w.h_kv, 0), dtype=torch.long, device=device)
    if w.n_clusters:
        starts = _cluster_starts(w, L, gen, device)[0]
        G = w.group
        qg = q[layer].to(device).float().reshape(w.h_kv, G * W, d)
        u = qg.mean(dim=1)
        u = u / u.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        shift = 1.5 * math.sqrt(d) * u                                       # [h_kv, d]
        span = torch.arange(w.cluster_len, device=device)
        rows = (starts[:, :, None] + span).reshape(w.h_kv, -1)               # [h_kv, n_clusters * 64]
        idx = rows[:, :, None].expand(-1, -1, d)
        k32.scatter_add_(1, idx, shift[:, None, :].expand(-1, rows.shape[1], -1).contiguous())
    k = k32.to(torch.bfloat16)
    del k32
    v = torch.randn((w.h_kv, n, d), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return k, v, starts


def _one_sequence(w: Workload, b: int, device):
    q = make_queries(w, b, device)
    n = w.prefix_lens[b] + w.window
    k = torch.empty((w.n_layers, w.h_kv, n, w.head_dim), device=device, dtype=torch.bfloat16)
    v = torch.empty_like(k)
    starts = []
    for layer in range(w.n_layers):
        k[layer], v[layer], st = make_layer(w, b, layer, q, device)
        starts.append(st)
    return q, k, v, torch.stack(starts)


def block_mask(w: Workload, device="cpu") -> tuple:
    """Seeded clustered block mask M[b, layer, h, i, j] (uint8) and per-sequence KV-block counts.

    The mask covers the last query chunk of each sequence (q_chunk tokens, so
    q_chunk / block query blocks) against ceil(L_b / block) KV blocks; entries
    at j >= n_kvblk[b] are zero.
    """
    gen = torch.Generator(device=device).manual_seed(w.seed ^ 0xB10C)
    n_qblk = w.q_chunk // w.block
    n_kv = [-(-L // w.block) for L in w.prefix_lens]
    nmax = max(n_kv)
    B, Lyr, H = w.batch, w.n_layers, w.h_q
    M = torch.zeros((B, Lyr, H, n_qblk, nmax), dtype=torch.uint8, device=device)
    jj = torch.arange(nmax, device=device)
    for b in range(B):
        nk = n_kv[b]
        target = w.mask_density * nk
        # expected run length 5; half the runs shared by all Q blocks, half drawn per Q block
        n_runs = max(1, int(round(target / 5.0)))
        n_shared = n_runs // 2
        n_own = n_runs - n_shared

        def runs(shape_prefix, count):
            st = torch.randint(0, nk, shape_prefix + (count,), generator=gen, device=device)
            ln = torch.randint(2, 9, shape_prefix + (count,), generator=gen, device=device)
            hit = (jj >= st[..., None]) & (jj < (st + ln)[..., None]) & (jj < nk)
            return hit.any(dim=-2)

        shared = runs((Lyr, H), n_shared)                     # [Lyr, H, nmax]
        own = runs((Lyr, H, n_qblk), n_own)                   # [Lyr, H, n_qblk, nmax]
        M[b] = (own | shared[:, :, None, :]).to(torch.uint8)
    return M, n_kv


def make_inputs(w: Workload, device="cpu", with_mask: Optional[bool] = None) -> Inputs:
    """All tensors of workload ``w`` on ``device`` (a torch device string)."""
    qs, ks, vs, cs = [], [], [], []
    for b in range(w.batch):
        q, k, v, c = _one_sequence(w, b, device)
        qs.append(q); ks.append(k); vs.append(v); cs.append(c)
    mask = n_kv = None
    if (w.block_union if with_mask is None else with_mask):
        mask, n_kv = block_mask(w, device)
    return Inputs(w, qs, ks, vs, cs, mask, n_kv)


def make_prompt_queries(w: Workload, b: int, device="cpu") -> torch.Tensor:
    """Queries of every prompt row of sequence b for the prefill: [n_layers, h_q, L_b + W, d] bf16.
    The last W rows are the observation-window queries of make_queries (same values); the prefix rows
    are drawn from their own stream."""
    L = w.prefix_lens[b]
    g = torch.Generator(device=device).manual_seed(w.seed * 1_000_003 + b * 10_007 + 0x51A7)
    pre = torch.randn((w.n_layers, w.h_q, L, w.head_dim), generator=g, device=device, dtype=torch.float32)
    return torch.cat([pre.to(torch.bfloat16), make_queries(w, b, device).to(device)], dim=2)


def make_decode_queries(w: Workload, n_q: int, device="cpu", seed_offset: int = 0) -> torch.Tensor:
    """Queries of n_q new tokens per head for attention over the selected cache:
    [batch, n_layers, h_q, n_q, d] bf16, N(0, 1)."""
    g = torch.Generator(device=device).manual_seed(w.seed * 7_919 + 0xDEC0DE + seed_offset)
    q = torch.randn((w.batch, w.n_layers, w.h_q, n_q, w.head_dim), generator=g, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16)


def random_scores(rows: int, n: int, seed: int, ties: bool = False, device="cpu") -> torch.Tensor:
    """Non-negative fp32 score rows for selection tests.

    With ``ties`` the values come from a small set of levels, so many equal
    scores straddle any k-th position and the index tie-break decides.
    """
    g = torch.Generator(device=device).manual_seed(seed)
    if ties:
        lv = torch.randint(0, 16, (rows, n), generator=g, device=device).float()
        return lv * 0.125
    return torch.rand((rows, n), generator=g, device=device, dtype=torch.float32)


def scaled(w: Workload, *, n_layers: Optional[int] = None, prefix_lens: Optional[Sequence[int]] = None,
           **kw) -> Workload:
    """A smaller copy of ``w`` (same structure) for tests the oracle finishes in seconds."""
    rep = dict(kw)
    if n_layers is not None:
        rep["n_layers"] = n_layers
        if w.layer_range is not None and "layer_range" not in kw:
            lo = min(w.layer_range[0], n_layers - 1)
            rep["layer_range"] = (lo, n_layers - 1)
    if prefix_lens is not None:
        rep["prefix_lens"] = tuple(int(x) for x in prefix_lens)
    return dataclasses.replace(w, **rep)
