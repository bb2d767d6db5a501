"""Plant plausible mistakes in fresh copies of the oracle: every one must fail some pin.

This shows the pins are strong enough that a dropped term, a wrong sign or
index, or a swapped operand anywhere in the oracle would be caught.
"""

import importlib.util
import inspect
import os

import numpy as np
import pytest

from tests import oracle_pins as pins

ORACLE_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "kvsel_oracle.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("kvsel_oracle_mutant", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _no_scale(o):
    o.window_logits = lambda q, k: q @ k.T


def _mask_off_by_one(o):
    def window_mask(L, W):
        return np.arange(L + W)[None, :] < L + np.arange(W)[:, None]
    o.window_mask = window_mask


def _prefix_only_softmax(o):
    def window_mask(L, W):
        return np.broadcast_to(np.arange(L + W)[None, :] < L, (W, L + W))
    o.window_mask = window_mask


def _mass_max_over_rows(o):
    o.column_mass = lambda p, L: p[:, :, :L].max(axis=1)


def _mass_includes_window_shift(o):
    o.column_mass = lambda p, L: p[:, :, 1:L + 1].sum(axis=1)


def _wrong_group_map(o):
    orig = o.group_scores

    def score_unit(q_layer, k_layer, g, G, L, mode, softmax=True):
        Hkv = q_layer.shape[0] // G
        return orig(o._f64(q_layer[g::Hkv]), o._f64(k_layer[g]), L, mode, softmax)
    o.score_unit = score_unit


def _reduce_swapped(o):
    orig = o.group_reduce
    o.group_reduce = lambda c, mode, W=1: orig(c, "max" if mode == "sum" else "sum" if mode == "max" else mode, W)


def _transposed_rows(o):
    """Window rows reversed against the mask (row j paired with the mask of row W-1-j)."""
    orig = o.window_probs

    def window_probs(q_group, k_head, L):
        return orig(q_group[:, ::-1], k_head, L)
    o.window_probs = window_probs


def _pool_radius(o):
    orig = o.max_pool
    o.max_pool = lambda s, k: orig(s, k + 2) if k > 1 else orig(s, k)


def _pool_one_sided(o):
    def max_pool(s, k):
        r = (k - 1) // 2
        out = s.copy()
        for off in range(1, r + 1):
            if off < s.shape[-1]:
                out[..., :-off] = np.maximum(out[..., :-off], s[..., off:])
        return out
    o.max_pool = max_pool


def _page_sum_for_max(o):
    orig = o.page_reduce
    o.page_reduce = lambda u, P, mode="max": orig(u, P, "sum")


def _tie_to_higher(o):
    def rank(scores):
        n = scores.shape[-1]
        return np.lexsort((-np.arange(n), -scores))
    o.rank = rank


def _rank_ascending(o):
    def rank(scores):
        n = scores.shape[-1]
        return np.lexsort((np.arange(n), scores))
    o.rank = rank


def _recency_off_by_one(o):
    orig = o.select_pages
    o.select_pages = lambda U, k, n_recent, L, W, P: orig(U, k, n_recent + 1, L, W, P)[1:]


def _no_l1(o):
    o.l1_normalise = lambda s: s


def _layer_range_exclusive(o):
    o.cross_layer_mean = lambda s, lo, hi: o.l1_normalise(s[lo:hi]).mean(axis=0)


def _union_wrong_group(o):
    def block_union(mask, h_kv, n_kv):
        out = []
        for g in range(h_kv):
            hit = np.zeros(n_kv, dtype=bool)
            for h in range(g, mask.shape[0], h_kv):
                hit |= (mask[h, :, :n_kv] != 0).any(axis=0)
            out.append(np.nonzero(hit)[0])
        return out
    o.block_union = block_union


def _union_first_qblock_only(o):
    def block_union(mask, h_kv, n_kv):
        G = mask.shape[0] // h_kv
        return [np.nonzero((mask[g * G:(g + 1) * G, 0, :n_kv] != 0).any(axis=0))[0] for g in range(h_kv)]
    o.block_union = block_union


def _gather_page_offset(o):
    orig = o.gather_rows
    o.gather_rows = lambda x, idx, page_size=1: orig(x, idx + (1 if page_size > 1 else 0), page_size)


def _logits_unscaled(o):
    def logit_mass(q_group, k_head, L):
        G, W, d = q_group.shape
        return (q_group.reshape(G * W, d) @ k_head[:L].T).reshape(G, W, L).sum(axis=1)
    o.logit_mass = logit_mass


def _logits_include_window_key(o):
    def logit_mass(q_group, k_head, L):
        G, W, d = q_group.shape
        z = o.window_logits(q_group.reshape(G * W, d), k_head[1:L + 1]).reshape(G, W, L)
        return z.sum(axis=1)
    o.logit_mass = logit_mass


def _mean_over_heads_only(o):
    orig = o.group_reduce
    o.group_reduce = lambda c, mode, W=1: c.sum(axis=0) / c.shape[0] if mode == "mean" else orig(c, mode, W)


def _head_sum_is_max(o):
    o.head_sum = lambda s: s.max(axis=-2)


def _avg_pool_counts_padding(o):
    def avg_pool(s, k):
        r = (k - 1) // 2
        n = s.shape[-1]
        tot = s.copy()
        for off in range(1, r + 1):
            if off < n:
                tot[..., :-off] += s[..., off:]
                tot[..., off:] += s[..., :-off]
        return tot / k
    o.avg_pool = avg_pool


def _layer_max_is_mean(o):
    o.layer_max = lambda s, lo, hi: s[lo:hi + 1].mean(axis=0)


def _keep_count_floor(o):
    o.keep_count = lambda r, L: int(min(L, max(0, np.floor(r * L))))


def _claa_buffer_short(o):
    orig = o.claa_sequence

    def claa_sequence(q, k, L, W, G, h_kv, defer, prune_layer, agg_window, keep_rate, pool_k=7, pool_kind="avg"):
        return orig(q, k, L, W, G, h_kv, defer, prune_layer, max(1, agg_window - 1), keep_rate, pool_k, pool_kind)
    o.claa_sequence = claa_sequence


def _attend_no_scale(o):
    def attend(q, k, v, rows):
        z = q @ k[rows].T
        p = np.exp(z - z.max(axis=-1, keepdims=True))
        return (p / p.sum(axis=-1, keepdims=True)) @ v[rows]
    o.attend = attend


def _table_rows_off_by_one(o):
    def table_rows(blocks, P, n_rows):
        rows = (np.asarray(blocks, np.int64)[:, None] * P + np.arange(1, P + 1)[None, :]).reshape(-1)
        return rows[rows < n_rows]
    o.table_rows = table_rows


def _prefill_not_causal(o):
    def prefill_attention(q, k, v):
        Hq, N, d = q.shape
        G = Hq // k.shape[0]
        out = np.zeros_like(q)
        lse = np.zeros((Hq, N))
        for h in range(Hq):
            z = o.window_logits(q[h], k[h // G])
            m = z.max(axis=-1, keepdims=True)
            e = np.exp(z - m)
            out[h] = (e / e.sum(-1, keepdims=True)) @ v[h // G]
            lse[h] = (m + np.log(e.sum(-1, keepdims=True)))[:, 0]
        return out, lse
    o.prefill_attention = prefill_attention


def _prefill_rows_sees_own_key_late(o):
    """Row i attends to keys t < i (its own key left out)."""
    orig = o.prefill_rows

    def prefill_rows(q, k, v, rows):
        out, lse = orig(q, k, v, [max(0, int(i) - 1) for i in rows])
        return out, lse
    o.prefill_rows = prefill_rows


def _rewrite_run_sequence(*edits):
    """A mutant that re-defines run_sequence from its own source with text edits (each must match once)."""
    def mutate(o):
        src = inspect.getsource(o.run_sequence)
        for old, new in edits:
            assert src.count(old) == 1, f"mutant pattern not found once: {old!r}"
            src = src.replace(old, new)
        exec(compile(src, o.__file__, "exec"), o.__dict__)
    return mutate


def _page_max_of_raw_scores(o):
    """Page scores taken from the unpooled token scores."""
    _rewrite_run_sequence(("U = page_reduce(u,", "U = page_reduce(raw,"))(o)


def _pool_after_page_max(o):
    """Page max first, then the pool over pages."""
    _rewrite_run_sequence(("U = page_reduce(u, w.page_size, w.page_reduce)",
                           "U = pool(page_reduce(raw, w.page_size, w.page_reduce), w.pool_k, kind)"))(o)


def _pool_before_l1_mean(o):
    """Cross-layer: each layer pooled before the L1 normalisation and the layer mean."""
    _rewrite_run_sequence(("s = cross_layer_mean(raw, lo, hi)", "s = cross_layer_mean(pool(raw, w.pool_k, kind), lo, hi)"),
                          ("u = pool(s, w.pool_k, kind)", "u = s"))(o)


def _run_layer_range_exclusive(o):
    """The last layer of the range left out inside the composition."""
    _rewrite_run_sequence(("cross_layer_mean(raw, lo, hi)", "cross_layer_mean(raw, lo, hi - 1)"))(o)


def _mean_over_every_layer(o):
    _rewrite_run_sequence(("cross_layer_mean(raw, lo, hi)", "cross_layer_mean(raw, 0, raw.shape[0] - 1)"))(o)


def _window_always_appended(o):
    _rewrite_run_sequence(('Wapp = W if getattr(w, "append_window", True) else 0', "Wapp = W"))(o)


def _head_sum_after_pool(o):
    _rewrite_run_sequence(("u = pool(head_sum(raw), w.pool_k, kind)", "u = head_sum(pool(raw, w.pool_k, kind))"))(o)


def _gather_first_layer_index(o):
    """Every layer's cache gathered with layer 0's selection."""
    _rewrite_run_sequence(('ii = out["idx"][i, g]', 'ii = out["idx"][0, g]'))(o)


def _pool_kind_ignored(o):
    _rewrite_run_sequence(('kind = getattr(w, "pool_type", "max")', 'kind = "max"'))(o)


MUTANTS = [_no_scale, _mask_off_by_one, _prefix_only_softmax, _mass_max_over_rows,
           _mass_includes_window_shift, _wrong_group_map, _reduce_swapped, _transposed_rows,
           _pool_radius, _pool_one_sided, _page_sum_for_max, _tie_to_higher, _rank_ascending,
           _recency_off_by_one, _no_l1, _layer_range_exclusive, _union_wrong_group,
           _union_first_qblock_only, _gather_page_offset, _logits_unscaled, _logits_include_window_key,
           _mean_over_heads_only, _head_sum_is_max, _avg_pool_counts_padding, _layer_max_is_mean,
           _keep_count_floor, _claa_buffer_short, _attend_no_scale, _table_rows_off_by_one,
           _prefill_not_causal, _page_max_of_raw_scores, _pool_after_page_max, _pool_before_l1_mean,
           _run_layer_range_exclusive, _mean_over_every_layer, _window_always_appended, _head_sum_after_pool,
           _gather_first_layer_index, _pool_kind_ignored, _prefill_rows_sees_own_key_late]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda m: m.__name__.strip("_"))
def test_mutant_is_caught(mutate):
    o = fresh_oracle()
    mutate(o)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(o)
        except Exception:          # an assertion, or a shape error the mistake causes
            failed.append(check.__name__)
    assert failed, f"no pin catches mutant {mutate.__name__}"
