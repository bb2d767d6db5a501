"""Thin ctypes binding of libkvsel.so (include/kvsel.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Functions keep the C names; tensors are passed by ``data_ptr()`` and
the stream is torch's current CUDA stream unless one is given.  A non-OK
status raises ``KvselError``.  If the library has not been built, importing
this module raises: there is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libkvsel.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(7)
REDUCE_SUM, REDUCE_MAX, REDUCE_MEAN = 0, 1, 2
POOL_MAX, POOL_AVG = 0, 1
SCORE_SOFTMAX, SCORE_LOGITS = 0, 1
LAYERS_EACH, LAYERS_L1_MEAN, LAYERS_MAX = 0, 1, 2
HEADS_EACH, HEADS_SUM = 0, 1
MAX_BATCH, MAX_WINDOW, MAX_ROWS, MAX_PAGE, WS_ALIGN = 128, 64, 256, 256, 256


class KvselError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32),
        ("h_q", ctypes.c_int32),
        ("h_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("prefix_lens", ctypes.POINTER(ctypes.c_int64)),
        ("group_reduce", ctypes.c_int32),
        ("pool_k", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("page_reduce", ctypes.c_int32),
        ("pool_type", ctypes.c_int32),
        ("score_mode", ctypes.c_int32),
        ("prefix_lens_dev", ctypes.c_void_p),
        ("prefix_len_max", ctypes.c_int64),
    ]


class ClaaParams(ctypes.Structure):
    _fields_ = [("defer", ctypes.c_int32), ("prune_layer", ctypes.c_int32), ("n_buffer", ctypes.c_int32),
                ("keep_rate", ctypes.c_double)]


class ClaaShape(ctypes.Structure):
    _fields_ = [("n_scored", ctypes.c_int32), ("buffer_lo", ctypes.c_int32), ("k", ctypes.c_int32),
                ("n_sel", ctypes.c_int32), ("ws_bytes", ctypes.c_size_t)]


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64), ("ms", ctypes.c_double)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with attention_kv_cache_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    D = P(Desc)
    sig = {
        "kvsel_workspace_size": (I32, [D, P(SZ)]),
        "kvsel_score": (I32, [D, VP, VP, VP, VP, VP, SZ, VP]),
        "kvsel_score_noalloc": (I32, [D, VP, VP, VP, VP, VP]),
        "kvsel_combine_layers": (I32, [D, VP, I32, I32, VP, VP, SZ, VP]),
        "kvsel_prefill_attention": (I32, [D, VP, VP, VP, VP, VP, VP, VP, VP, VP]),
        "kvsel_score_from_lse": (I32, [D, VP, VP, VP, VP, VP, VP, SZ, VP]),
        "kvsel_aggregate": (I32, [D, VP, I32, I32, I32, I32, VP, VP, SZ, VP]),
        "kvsel_select": (I32, [D, VP, I32, I32, I32, I32, VP, VP, SZ, VP]),
        "kvsel_topk": (I32, [D, VP, I32, I32, I32, VP, VP, SZ, VP]),
        "kvsel_compact": (I32, [D, VP, VP, VP, I32, I32, VP, VP, VP, VP]),
        "kvsel_compact_layers": (I32, [D, VP, VP, VP, I32, I32, I32, I32, I32, VP, VP, VP, VP]),
        "kvsel_pagetable": (I32, [D, VP, I32, I32, VP, VP, VP, VP, SZ, VP]),
        "kvsel_claa_shape": (I32, [D, P(ClaaParams), P(ClaaShape)]),
        "kvsel_claa_select": (I32, [D, P(ClaaParams), VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP, SZ, VP]),
        "kvsel_attend_workspace_size": (I32, [D, I32, I32, I32, P(SZ)]),
        "kvsel_attend": (I32, [D, VP, I32, VP, VP, VP, VP, I32, I32, I32, VP, VP, SZ, VP]),
        "kvsel_read_device_error": (I32, [VP, VP]),
        "kvsel_noalloc_read_device_error": (I32, [VP]),
        "kvsel_selftest_bounded_wait": (I32, [VP, ctypes.c_uint32, I32, VP]),
        "kvsel_status_string": (ctypes.c_char_p, [I32]),
        "kvsel_version": (ctypes.c_char_p, []),
        "kvsel_trace_enable": (None, [I32]),
        "kvsel_trace_read": (I32, [P(TraceEntry), I32, P(I32)]),
        "kvsel_launch_count": (I64, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()
EXPORTED = ("kvsel_workspace_size", "kvsel_score", "kvsel_score_noalloc", "kvsel_prefill_attention",
            "kvsel_score_from_lse", "kvsel_combine_layers",
            "kvsel_aggregate", "kvsel_select", "kvsel_topk", "kvsel_compact", "kvsel_compact_layers",
            "kvsel_pagetable", "kvsel_claa_shape", "kvsel_claa_select", "kvsel_attend_workspace_size", "kvsel_attend", "kvsel_read_device_error", "kvsel_noalloc_read_device_error", "kvsel_selftest_bounded_wait", "kvsel_status_string",
            "kvsel_version", "kvsel_trace_enable", "kvsel_trace_read", "kvsel_launch_count")


def status_string(status: int) -> str:
    return _lib.kvsel_status_string(status).decode()


def version() -> str:
    return _lib.kvsel_version().decode()


def _check(status: int, what: str):
    if status != OK:
        raise KvselError(status, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_desc(*, n_layers: int, h_q: int, h_kv: int, head_dim: int, window: int,
              prefix_lens: Optional[Sequence[int]] = None, group_reduce: int = REDUCE_SUM, pool_k: int = 7,
              page_size: int = 1, page_reduce: int = REDUCE_MAX, pool_type: int = POOL_MAX,
              score_mode: int = SCORE_SOFTMAX, prefix_lens_dev=None, prefix_len_max: int = 0) -> Desc:
    """A descriptor; it keeps its own host copy of prefix_lens (or a reference to the device tensor
    ``prefix_lens_dev``, int64 on the GPU, with its bound ``prefix_len_max``) alive."""
    if prefix_lens_dev is not None:
        if prefix_lens is not None:
            raise ValueError("give prefix_lens or prefix_lens_dev, not both")
        d = Desc(n_layers, h_q, h_kv, head_dim, window, int(prefix_lens_dev.numel()), None, group_reduce,
                 pool_k, page_size, page_reduce, pool_type, score_mode, _ptr(prefix_lens_dev), int(prefix_len_max))
        d._lens = prefix_lens_dev
        return d
    lens = (ctypes.c_int64 * len(prefix_lens))(*[int(x) for x in prefix_lens])
    d = Desc(n_layers, h_q, h_kv, head_dim, window, len(prefix_lens), lens, group_reduce, pool_k,
             page_size, page_reduce, pool_type, score_mode, None, 0)
    d._lens = lens
    return d


def kvsel_workspace_size(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.kvsel_workspace_size(ctypes.byref(desc), ctypes.byref(n)), "kvsel_workspace_size")
    return n.value


def kvsel_score(desc, q, k, scores, page_scores, ws, ws_bytes: Optional[int] = None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_score(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(scores), _ptr(page_scores), _ptr(ws),
                            nb, _stream(stream)), "kvsel_score")


def kvsel_score_noalloc(desc, q, k, scores, page_scores, stream=None):
    """kvsel_score with the library's built-in scratch (no workspace argument, nothing allocated)."""
    _check(_lib.kvsel_score_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(scores), _ptr(page_scores),
                                    _stream(stream)), "kvsel_score_noalloc")


NOALLOC_SCRATCH_BYTES = 32 << 20


def kvsel_prefill_attention(desc, q, k, v, o, lse, lse_win, q_win, ws=None, stream=None):
    _check(_lib.kvsel_prefill_attention(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                        _ptr(lse_win), _ptr(q_win), _ptr(ws), _stream(stream)),
           "kvsel_prefill_attention")


def kvsel_score_from_lse(desc, q_win, k, lse_win, scores, page_scores, ws, ws_bytes=None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_score_from_lse(ctypes.byref(desc), _ptr(q_win), _ptr(k), _ptr(lse_win), _ptr(scores),
                                     _ptr(page_scores), _ptr(ws), nb, _stream(stream)), "kvsel_score_from_lse")


def kvsel_combine_layers(desc, scores, layer_lo: int, layer_hi: int, combined, ws, ws_bytes=None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_combine_layers(ctypes.byref(desc), _ptr(scores), layer_lo, layer_hi, _ptr(combined),
                                     _ptr(ws), nb, _stream(stream)), "kvsel_combine_layers")


def kvsel_aggregate(desc, scores, layer_lo: int, layer_hi: int, layer_op: int, head_op: int, out, ws,
                    ws_bytes=None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_aggregate(ctypes.byref(desc), _ptr(scores), layer_lo, layer_hi, layer_op, head_op, _ptr(out),
                                _ptr(ws), nb, _stream(stream)), "kvsel_aggregate")


def kvsel_select(desc, scores, rows: int, k: int, n_recent: int, append_window: bool, idx_out, ws, ws_bytes=None,
                 stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_select(ctypes.byref(desc), _ptr(scores), rows, k, n_recent, 1 if append_window else 0,
                             _ptr(idx_out), _ptr(ws), nb, _stream(stream)), "kvsel_select")


def kvsel_topk(desc, scores, layers: int, k: int, n_recent: int, idx_out, ws, ws_bytes=None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_topk(ctypes.byref(desc), _ptr(scores), layers, k, n_recent, _ptr(idx_out), _ptr(ws), nb,
                           _stream(stream)), "kvsel_topk")


def kvsel_compact(desc, k, v, idx, idx_layers: int, n_sel: int, k_out, v_out, ws=None, stream=None):
    _check(_lib.kvsel_compact(ctypes.byref(desc), _ptr(k), _ptr(v), _ptr(idx), idx_layers, n_sel, _ptr(k_out),
                              _ptr(v_out), _ptr(ws), _stream(stream)), "kvsel_compact")


def kvsel_compact_layers(desc, k, v, idx, idx_layers: int, idx_heads: int, layer_lo: int, n_layers_out: int,
                         n_sel: int, k_out, v_out, ws=None, stream=None):
    _check(_lib.kvsel_compact_layers(ctypes.byref(desc), _ptr(k), _ptr(v), _ptr(idx), idx_layers, idx_heads,
                                     layer_lo, n_layers_out, n_sel, _ptr(k_out), _ptr(v_out), _ptr(ws),
                                     _stream(stream)), "kvsel_compact_layers")


def kvsel_pagetable(desc, mask, n_qblk: int, n_kvblk_max: int, n_kvblk: Sequence[int], kv_indptr, kv_indices,
                    ws, ws_bytes=None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    if hasattr(n_kvblk, "data_ptr"):            # int32 device tensor (descriptor with device lengths)
        nk = _ptr(n_kvblk)
    else:
        arr = (ctypes.c_int32 * len(n_kvblk))(*[int(x) for x in n_kvblk])
        nk = ctypes.cast(arr, ctypes.c_void_p)
    _check(_lib.kvsel_pagetable(ctypes.byref(desc), _ptr(mask), n_qblk, n_kvblk_max, nk, _ptr(kv_indptr),
                                _ptr(kv_indices), _ptr(ws), nb, _stream(stream)), "kvsel_pagetable")


def kvsel_claa_shape(desc, params: ClaaParams) -> ClaaShape:
    out = ClaaShape()
    _check(_lib.kvsel_claa_shape(ctypes.byref(desc), ctypes.byref(params), ctypes.byref(out)), "kvsel_claa_shape")
    return out


def kvsel_claa_select(desc, params: ClaaParams, q, k, v, scores, layer_scores, prune_scores, idx, prune_idx, k_out,
                      v_out, ws, ws_bytes=None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_claa_select(ctypes.byref(desc), ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(scores),
                                  _ptr(layer_scores), _ptr(prune_scores), _ptr(idx), _ptr(prune_idx), _ptr(k_out),
                                  _ptr(v_out), _ptr(ws), nb, _stream(stream)), "kvsel_claa_select")


def kvsel_attend_workspace_size(desc, n_q: int, block: int, max_blocks: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.kvsel_attend_workspace_size(ctypes.byref(desc), n_q, block, max_blocks, ctypes.byref(n)),
           "kvsel_attend_workspace_size")
    return n.value


def kvsel_attend(desc, q, n_q: int, k, v, kv_indptr, kv_indices, n_per_row: int, block: int, max_blocks: int, o,
                 ws, ws_bytes=None, stream=None):
    nb = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(_lib.kvsel_attend(ctypes.byref(desc), _ptr(q), n_q, _ptr(k), _ptr(v), _ptr(kv_indptr), _ptr(kv_indices),
                             n_per_row, block, max_blocks, _ptr(o), _ptr(ws), nb, _stream(stream)), "kvsel_attend")


def kvsel_read_device_error(ws, stream=None) -> int:
    """Status recorded by the device in the workspace's error word (clears it)."""
    return _lib.kvsel_read_device_error(_ptr(ws), _stream(stream))


def kvsel_noalloc_read_device_error(stream=None) -> int:
    """Status the device recorded during the last kvsel_score_noalloc call on the current device (clears it)."""
    return _lib.kvsel_noalloc_read_device_error(_stream(stream))


def kvsel_selftest_bounded_wait(ws, polls: int, arrive: bool, stream=None):
    _check(_lib.kvsel_selftest_bounded_wait(_ptr(ws), polls, 1 if arrive else 0, _stream(stream)),
           "kvsel_selftest_bounded_wait")


def kvsel_trace_enable(on: bool):
    _lib.kvsel_trace_enable(1 if on else 0)


def kvsel_trace_read() -> dict:
    n = ctypes.c_int32(0)
    buf = (TraceEntry * 64)()
    _check(_lib.kvsel_trace_read(buf, 64, ctypes.byref(n)), "kvsel_trace_read")
    return {buf[i].name.decode(): (buf[i].launches, buf[i].ms) for i in range(min(n.value, 64))}


def kvsel_launch_count() -> int:
    return _lib.kvsel_launch_count()


def raw_call(name: str, *args) -> int:
    """The C function itself (status returned, nothing raised), for argument-check tests."""
    return getattr(_lib, name)(*args)
