"""Comparison rules between the CUDA path and the fp64 oracle.

* fp32 scores: |gpu - oracle| <= 1e-3 * |oracle| + 1e-6 element by element.
  Pre-softmax (logit) scores are signed sums that can cancel to near zero, so
  a relative bound says little where they do; their absolute term adds a
  per-element bound of the fp32 dot-product error instead.  The fp32
  accumulation of one d-term dot product of bf16 values (the products are
  exact) is off by about sqrt(d) * 2^-24 * sum_c |q_c k_c| (random-walk
  rounding), which the 1 / sqrt(d) scale turns into 2^-24 * sum_c |q_c k_c|
  per logit; summed over the rows a score adds up, that is
  B[t] = 2^-24 * sum_r sum_c |q_rc k_tc|, computed in fp64 from the inputs
  (``logit_error_scale``).  The test allows LOGIT_SAFETY * B[t], carried
  through pooling (the largest B in the pool window) and the head sum.
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


LOGIT_SAFETY = 2.0
U32 = 2.0 ** -24

# Largest |gpu - oracle| / B seen by assert_scores_close with a bound (reported by the logit tests).
WORST_LOGIT_RATIO = {"ratio": 0.0, "what": ""}


def _np64(x):
    if hasattr(x, "detach"):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, np.float64)


def logit_error_scale(q_layer, k_layer, G: int, L: int) -> np.ndarray:
    """B [H_kv, L]: 2^-24 * sum over the G * W rows r of each group and the d channels c of |q_rc k_tc|.

    q_layer [H_q, W, d], k_layer [H_kv, L + W, d] (bf16 tensors or arrays), in fp64.
    """
    q = np.abs(_np64(q_layer))
    k = np.abs(_np64(k_layer))
    d = q.shape[-1]
    out = []
    for g in range(k.shape[0]):
        colsum = q[g * G:(g + 1) * G].reshape(-1, d).sum(axis=0)     # sum_r |q_rc|
        out.append(U32 * (k[g, :L] @ colsum))
    return np.stack(out)


def pooled_bound(b: np.ndarray, pool_k: int) -> np.ndarray:
    """The largest bound over each pool window (last axis): a pooled value's error is at most that."""
    r = (pool_k - 1) // 2
    out = b.copy()
    for off in range(1, r + 1):
        if off >= b.shape[-1]:
            break
        out[..., :-off] = np.maximum(out[..., :-off], b[..., off:])
        out[..., off:] = np.maximum(out[..., off:], b[..., :-off])
    return out


def assert_scores_close(gpu, ref, what="scores", bound=None):
    """|gpu - oracle| <= RTOL |oracle| + ATOL (+ LOGIT_SAFETY * bound for pre-softmax scores)."""
    g = _np64(gpu)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    atol = ATOL if bound is None else ATOL + LOGIT_SAFETY * np.broadcast_to(np.asarray(bound, np.float64), r.shape)
    err = np.abs(g - r)
    if bound is not None:
        ratio = float((err / np.maximum(np.broadcast_to(bound, r.shape), 1e-300)).max())
        if ratio > WORST_LOGIT_RATIO["ratio"]:
            WORST_LOGIT_RATIO.update(ratio=ratio, what=what)
    bad = err > RTOL * np.abs(r) + atol
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
