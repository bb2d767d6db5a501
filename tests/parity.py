"""Comparison rules between the CUDA path and the fp64 oracle.

* fp32 scores: |gpu - oracle| <= 1e-3 * |oracle| + 1e-6 element by element.
  Pre-softmax (logit) scores are signed sums that can cancel to near zero, so
  their absolute term scales with the row: 1e-4 * RMS of the oracle row.  (The
  fp32 accumulation of one 128-term bf16 dot product is off by about
  sqrt(d) * 2^-24 * sum |q_i k_i| ~ 1e-6 of a logit of order one.)
* Selected sets: equal, except that an index may be swapped for another when
  the oracle score of each lies within 1e-5 (relative) of the oracle's k-th
  score — a near tie that fp32 and fp64 may order differently.  The appended
  recency / window part must be identical, and the GPU list must be strictly
  ascending.
* Integer, index and byte outputs (page tables, gathered rows): bit-exact.
"""

from __future__ import annotations

import numpy as np
import torch

RTOL, ATOL, TIE_RTOL = 1e-3, 1e-6, 1e-5


LOGIT_ATOL_RMS = 1e-4


def assert_scores_close(gpu, ref, what="scores", signed=False):
    """signed=True for pre-softmax (logit) scores: the absolute term is 1e-4 * RMS of each last-axis row."""
    g = gpu.detach().float().cpu().double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    atol = LOGIT_ATOL_RMS * np.sqrt((r * r).mean(axis=-1, keepdims=True)) if signed else ATOL
    bad = np.abs(g - r) > RTOL * np.abs(r) + atol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu {g[tuple(i)]!r} oracle {r[tuple(i)]!r}")


def assert_selection_equivalent(gpu_sel, ref_sel, ref_scores, k, what="selection"):
    """gpu_sel / ref_sel: 1-D int arrays (k selected entries, then the fixed tail)."""
    g = np.asarray(gpu_sel, np.int64)
    r = np.asarray(ref_sel, np.int64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    np.testing.assert_array_equal(g[k:], r[k:], err_msg=f"{what}: appended part differs")
    assert np.all(np.diff(g[:k]) > 0), f"{what}: selection not strictly ascending"
    if k == 0:
        return
    s = np.asarray(ref_scores, np.float64)
    gs, rs = set(g[:k].tolist()), set(r[:k].tolist())
    if gs == rs:
        return
    kth = s[list(rs)].min()
    for x in gs ^ rs:
        assert 0 <= x < len(s), f"{what}: index {x} out of range"
        assert abs(s[x] - kth) <= TIE_RTOL * abs(kth), \
            f"{what}: index {x} (oracle score {s[x]!r}) differs but k-th score is {kth!r}"


def gathered_rows_match(k_out, k_in, sel, page_size, n_keys):
    """Rows of k_out ([n_sel * P, d] bf16) equal k_in ([n_keys, d]) at sel (bytes), zero past n_keys."""
    ko = k_out.cpu().view(torch.int16)
    ki = k_in.cpu().view(torch.int16)
    sel = torch.as_tensor(np.asarray(sel, np.int64))
    if page_size == 1:
        rows = sel
    else:
        rows = (sel[:, None] * page_size + torch.arange(page_size)[None, :]).reshape(-1)
    want = torch.zeros_like(ko)
    ok = rows < n_keys
    want[ok] = ki[rows[ok]]
    return torch.equal(ko, want)
