"""The C-ABI library loads, exports every declared symbol and rejects bad arguments on the host (no GPU)."""

import ctypes
import os
import re

import pytest

from attention_kv_cache_gb300 import kvsel as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "kvsel.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"KVSEL_API[^;(]*?\b(kvsel_\w+)\s*\(", text, flags=re.S)))


def test_header_declares_the_four_operations():
    names = declared_symbols()
    for op in ("kvsel_score", "kvsel_topk", "kvsel_compact", "kvsel_pagetable", "kvsel_combine_layers"):
        assert op in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(K.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(K.EXPORTED)
    assert "sm_103a" in K.version()
    assert K.status_string(K.ERR_WORKSPACE).startswith("workspace")


def _desc(**kw):
    base = dict(n_layers=2, h_q=8, h_kv=2, head_dim=128, window=32, prefix_lens=[1000])
    base.update(kw)
    return K.make_desc(**base)


def test_workspace_size_grows_with_length():
    a = K.kvsel_workspace_size(_desc(prefix_lens=[1000]))
    b = K.kvsel_workspace_size(_desc(prefix_lens=[100000]))
    c = K.kvsel_workspace_size(_desc(prefix_lens=[1000, 5000, 70000]))
    assert 0 < a < b and c > a and a % K.WS_ALIGN == 0


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), K.ERR_UNSUPPORTED),
    (dict(h_q=6, h_kv=4), K.ERR_INVALID_ARG),
    (dict(window=0), K.ERR_INVALID_ARG),
    (dict(window=65), K.ERR_INVALID_ARG),
    (dict(h_q=32, h_kv=2, window=32), K.ERR_UNSUPPORTED),      # 16 heads x 32 rows > 256
    (dict(pool_k=4), K.ERR_INVALID_ARG),
    (dict(pool_k=65), K.ERR_INVALID_ARG),
    (dict(page_size=0), K.ERR_INVALID_ARG),
    (dict(page_size=512), K.ERR_INVALID_ARG),
    (dict(prefix_lens=[0]), K.ERR_INVALID_ARG),
    (dict(prefix_lens=[2 ** 31]), K.ERR_INVALID_ARG),
    (dict(prefix_lens=[10] * 129), K.ERR_INVALID_ARG),
    (dict(group_reduce=3), K.ERR_INVALID_ARG),
    (dict(pool_type=2), K.ERR_INVALID_ARG),
    (dict(score_mode=2), K.ERR_INVALID_ARG),
    (dict(page_reduce=2), K.ERR_INVALID_ARG),
])
def test_bad_descriptor_rejected(kw, status):
    d = _desc(**kw)
    n = ctypes.c_size_t(0)
    assert K.raw_call("kvsel_workspace_size", ctypes.byref(d), ctypes.byref(n)) == status
    # the same check runs before any launch in every entry point (null stream: nothing is touched)
    assert K.raw_call("kvsel_score", ctypes.byref(d), 16, 16, 16, 16, 256, 1 << 40, None) == status


@pytest.mark.parametrize("h_q,h_kv,window,reduce", [
    (8, 2, 24, K.REDUCE_MAX),      # heads padded to 32 rows: 128 tile rows
    (8, 2, 40, K.REDUCE_MAX),      # padded to 64 rows: 256 tile rows
    (20, 2, 24, K.REDUCE_MAX),     # 240 rows, 320 once padded: the CUDA-core kernels
    (64, 2, 8, K.REDUCE_SUM),      # 256 rows of 8-row heads
    (2, 2, 64, K.REDUCE_MEAN),     # one head of the widest window
])
def test_supported_group_shapes_accepted(h_q, h_kv, window, reduce):
    """Every shape within (h_q / h_kv) W <= 256 has a kernel, whatever its padding."""
    d = _desc(h_q=h_q, h_kv=h_kv, window=window, group_reduce=reduce)
    assert K.kvsel_workspace_size(d) > 0


def test_null_and_misaligned_pointers_rejected():
    d = _desc()
    ws = K.kvsel_workspace_size(d)
    assert K.raw_call("kvsel_score", ctypes.byref(d), None, 16, 16, None, 256, ws, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_score", ctypes.byref(d), 8, 16, 16, None, 256, ws, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_score", ctypes.byref(d), 16, 16, 16, None, None, ws, None) == K.ERR_WORKSPACE
    assert K.raw_call("kvsel_score", ctypes.byref(d), 16, 16, 16, None, 128, ws, None) == K.ERR_WORKSPACE
    assert K.raw_call("kvsel_score", ctypes.byref(d), 16, 16, 16, None, 256, ws - 1, None) == K.ERR_WORKSPACE
    dp = _desc(page_size=16)
    assert K.raw_call("kvsel_score", ctypes.byref(dp), 16, 16, 16, None, 256, 1 << 40, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_compact", ctypes.byref(d), 16, 16, 16, 1, 10, 16, 8, None, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_compact", ctypes.byref(d), 16, 16, 16, 3, 10, 16, 16, None, None) == K.ERR_INVALID_ARG


def test_selection_arguments_rejected():
    d = _desc(prefix_lens=[100])
    big = 1 << 40
    assert K.raw_call("kvsel_topk", ctypes.byref(d), 16, 2, 101, 0, 16, 256, big, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_topk", ctypes.byref(d), 16, 2, 5, 1, 16, 256, big, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_topk", ctypes.byref(d), 16, 3, 5, 0, 16, 256, big, None) == K.ERR_INVALID_ARG
    dp = _desc(prefix_lens=[100], page_size=16)          # 7 pages, the last one partial
    assert K.raw_call("kvsel_topk", ctypes.byref(dp), 16, 2, 3, 0, 16, 256, big, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_topk", ctypes.byref(dp), 16, 2, 7, 1, 16, 256, big, None) == K.ERR_INVALID_ARG
    dw = _desc(prefix_lens=[96], page_size=16, window=24)  # window not a whole number of pages
    assert K.raw_call("kvsel_topk", ctypes.byref(dw), 16, 2, 2, 1, 16, 256, big, None) == K.ERR_UNSUPPORTED
    nk = (ctypes.c_int32 * 1)(9)
    assert K.raw_call("kvsel_pagetable", ctypes.byref(d), 16, 4, 8, nk, 16, 16, 256, big, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_combine_layers", ctypes.byref(d), 16, 1, 2, 16, 256, big, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_selftest_bounded_wait", None, 10, 0, None) == K.ERR_WORKSPACE
    assert K.raw_call("kvsel_selftest_bounded_wait", 256, 0, 0, None) == K.ERR_INVALID_ARG


def test_new_entry_arguments_rejected():
    """kvsel_aggregate / kvsel_select / kvsel_compact_layers check their arguments before any launch."""
    d = _desc(prefix_lens=[100])
    big = 1 << 40
    agg = lambda lo, hi, lop, hop: K.raw_call("kvsel_aggregate", ctypes.byref(d), 16, lo, hi, lop, hop, 16, 256,
                                              big, None)
    assert agg(0, 2, K.LAYERS_MAX, K.HEADS_SUM) == K.ERR_INVALID_ARG        # layer beyond n_layers
    assert agg(1, 0, K.LAYERS_MAX, K.HEADS_SUM) == K.ERR_INVALID_ARG        # empty range
    assert agg(0, 1, 3, K.HEADS_SUM) == K.ERR_INVALID_ARG
    assert agg(0, 1, K.LAYERS_EACH, 2) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_aggregate", ctypes.byref(d), None, 0, 1, 0, 0, 16, 256, big, None) == K.ERR_INVALID_ARG
    sel = lambda rows, k, nr, app: K.raw_call("kvsel_select", ctypes.byref(d), 16, rows, k, nr, app, 16, 256, big,
                                              None)
    assert sel(0, 5, 0, 1) == K.ERR_INVALID_ARG
    assert sel(3, 101, 0, 0) == K.ERR_INVALID_ARG
    assert sel(3, 5, 1, 1) == K.ERR_INVALID_ARG                             # recency is a page-mode option
    cl = lambda il, ih, lo, n: K.raw_call("kvsel_compact_layers", ctypes.byref(d), 16, 16, 16, il, ih, lo, n, 10,
                                          16, 16, None, None)
    assert cl(1, 1, 1, 2) == K.ERR_INVALID_ARG                              # layers 1..2 of 2
    assert cl(2, 1, 1, 1) == K.ERR_INVALID_ARG                              # idx rows != compacted layers
    assert cl(1, 3, 0, 2) == K.ERR_INVALID_ARG                              # idx heads neither 1 nor h_kv
    assert K.raw_call("kvsel_compact_layers", ctypes.byref(d), 16, 16, 16, 1, 1, 0, 2, 10, 8, 16, None,
                      None) == K.ERR_INVALID_ARG                            # misaligned output


def _dev_desc(lmax, **kw):
    """A descriptor whose lengths are 'on the device' (a fake address: nothing is dereferenced on the host)."""
    d = _desc(**kw)
    d.prefix_lens = None
    d.prefix_lens_dev = 256
    d.prefix_len_max = lmax
    return d


def test_device_length_descriptor_checks():
    n = ctypes.c_size_t(0)
    d = _dev_desc(5000)
    assert K.raw_call("kvsel_workspace_size", ctypes.byref(d), ctypes.byref(n)) == K.OK
    # the workspace is sized for the bound
    assert n.value == K.kvsel_workspace_size(_desc(prefix_lens=[5000]))
    both = _dev_desc(5000)
    both.prefix_lens = _desc().prefix_lens
    assert K.raw_call("kvsel_workspace_size", ctypes.byref(both), ctypes.byref(n)) == K.ERR_INVALID_ARG
    neither = _desc()
    neither.prefix_lens = None
    assert K.raw_call("kvsel_workspace_size", ctypes.byref(neither), ctypes.byref(n)) == K.ERR_INVALID_ARG
    for lmax in (0, 2 ** 31):
        assert K.raw_call("kvsel_workspace_size", ctypes.byref(_dev_desc(lmax)), ctypes.byref(n)) == K.ERR_INVALID_ARG
    big = 1 << 40
    # checks against the bound still run on the host: k above it, recency beyond its pages
    assert K.raw_call("kvsel_topk", ctypes.byref(_dev_desc(100)), 16, 2, 101, 0, 16, 256, big, None) == K.ERR_INVALID_ARG
    assert K.raw_call("kvsel_topk", ctypes.byref(_dev_desc(100, page_size=16)), 16, 2, 7, 1, 16, 256, big,
                      None) == K.ERR_INVALID_ARG
    # every call needs a workspace: it holds the table built on the device
    assert K.raw_call("kvsel_compact", ctypes.byref(_dev_desc(100)), 16, 16, 16, 1, 10, 16, 16, None,
                      None) == K.ERR_WORKSPACE
    # the prefill takes host lengths only
    assert K.raw_call("kvsel_prefill_attention", ctypes.byref(_dev_desc(100)), 16, 16, 16, 16, None, 16, 16, 256,
                      None) == K.ERR_UNSUPPORTED


def test_claa_shape_matches_the_oracle_schedule():
    """kvsel_claa_shape's keep count and buffer follow CLAA's schedule as the oracle writes it (host only)."""
    from oracle import kvsel_oracle as O
    for rate, L in ((0.2, 32768), (0.1, 30), (0.25, 10), (0.15, 10), (1.0, 7), (0.0, 5), (0.5, 1), (0.4, 3),
                    (0.1, 32768), (0.33, 1001)):
        d = _desc(n_layers=16, h_q=32, h_kv=8, window=8, prefix_lens=[L], pool_k=7, pool_type=K.POOL_AVG)
        for m, lp, n in ((4, 15, 4), (2, 6, 3), (3, 4, 4), (0, 0, 1)):
            sh = K.kvsel_claa_shape(d, K.ClaaParams(m, lp, n, rate))
            assert sh.k == O.keep_count(rate, L), (rate, L, sh.k)
            assert sh.n_sel == sh.k + 8
            assert sh.n_scored == lp - m + 1
            assert sh.buffer_lo == max(m, lp - n + 1)
            assert sh.ws_bytes >= K.kvsel_workspace_size(d)
    d = _desc(n_layers=16, prefix_lens=[100])
    bad = [K.ClaaParams(5, 4, 4, 0.2), K.ClaaParams(4, 16, 4, 0.2), K.ClaaParams(4, 15, 0, 0.2),
           K.ClaaParams(4, 15, 4, 1.5), K.ClaaParams(-1, 15, 4, 0.2)]
    out = K.ClaaShape()
    for p in bad:
        assert K.raw_call("kvsel_claa_shape", ctypes.byref(d), ctypes.byref(p), ctypes.byref(out)) == K.ERR_INVALID_ARG
    p = K.ClaaParams(4, 15, 4, 0.2)
    assert K.raw_call("kvsel_claa_shape", ctypes.byref(_desc(n_layers=16, prefix_lens=[100, 200])), ctypes.byref(p),
                      ctypes.byref(out)) == K.ERR_UNSUPPORTED
    assert K.raw_call("kvsel_claa_shape", ctypes.byref(_desc(n_layers=16, prefix_lens=[100], group_reduce=K.REDUCE_MAX)),
                      ctypes.byref(p), ctypes.byref(out)) == K.ERR_INVALID_ARG
