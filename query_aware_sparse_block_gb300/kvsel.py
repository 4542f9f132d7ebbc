"""ctypes binding of libkvsel.so (argument marshalling only).

Every function here forwards torch tensors' device pointers and the current
CUDA stream to the C entry point of the same name in ``include/kvsel.h``; all
compute runs in the library's CUDA kernels. There is no fallback: if the
library is missing or a call fails, a ``KvselError`` is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvsel.so")

KVSEL_OK = 0
KVSEL_ERR_INVALID_ARG = 1
KVSEL_ERR_CUDA = 2
KVSEL_ERR_BOUNDS = 3
KVSEL_ERR_TIMEOUT = 4
KVSEL_ERR_UNSUPPORTED = 5
KVSEL_ERR_WORKSPACE = 6

KVSEL_SUMMARY_FULL = 0
KVSEL_SUMMARY_APPEND = 1
KVSEL_KV_PAGED = 0
KVSEL_KV_STAGED = 1
KVSEL_KV_HOST = 2
KVSEL_KV_HOST_DIRECT = 3
KVSEL_WS_SCORE_TOPK = 0
KVSEL_WS_SPARSE_DECODE = 1
KVSEL_WS_CACHE_FETCH = 2
KVSEL_SCORE_PATH_AUTO = 0
KVSEL_SCORE_PATH_TWO_GRID = 1
KVSEL_SCORE_PATH_CLUSTER = 2

_STATUS = {1: "INVALID_ARG", 2: "CUDA", 3: "BOUNDS", 4: "TIMEOUT", 5: "UNSUPPORTED", 6: "WORKSPACE"}


class KvselError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        super().__init__(f"{where}: KVSEL_ERR_{_STATUS.get(code, code)} {detail}".rstrip())


class kvsel_problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_qheads", ctypes.c_int32),
                ("n_kvheads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("k_max", ctypes.c_int32)]


class kvsel_append_in(ctypes.Structure):
    _fields_ = [("kv_pages", ctypes.c_void_p), ("n_pages", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("append_pos", ctypes.c_void_p),
                ("new_k", ctypes.c_void_p), ("new_v", ctypes.c_void_p),
                ("summaries", ctypes.c_void_p), ("open_acc", ctypes.c_void_p)]


class kvsel_window(ctypes.Structure):
    _fields_ = [("n_sink", ctypes.c_int32), ("n_recent", ctypes.c_int32)]


class kvsel_block_cache(ctypes.Structure):
    _fields_ = [("slots", ctypes.c_int32), ("pool", ctypes.c_void_p), ("page_of", ctypes.c_void_p),
                ("block_in", ctypes.c_void_p), ("last_use", ctypes.c_void_p)]


class kvsel_kv_src(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("staging_slots", ctypes.c_int32),
                ("kv_pages", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("n_pages", ctypes.c_int64),
                ("staging", ctypes.c_void_p), ("host_kv", ctypes.c_void_p),
                ("host_blocks", ctypes.c_int32), ("fetch_ctas", ctypes.c_int32)]


class kvsel_budget_in(ctypes.Structure):
    _fields_ = [("block_size", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("elem_bytes", ctypes.c_int32),
                ("hidden", ctypes.c_int64), ("n_blocks", ctypes.c_int64),
                ("h2d_bytes_per_s", ctypes.c_double), ("recompute_flop_per_s", ctypes.c_double),
                ("kappa", ctypes.c_double), ("keep_floor", ctypes.c_double),
                ("gamma", ctypes.c_double), ("tau_s", ctypes.c_double),
                ("keep_override", ctypes.c_double)]


class kvsel_budget_out(ctypes.Structure):
    _fields_ = [("c_copy_s", ctypes.c_double), ("c_rec_s", ctypes.c_double),
                ("r_model", ctypes.c_double), ("r", ctypes.c_double), ("k", ctypes.c_int64),
                ("tau_rel", ctypes.c_double), ("dense", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "kvsel_build_summaries": (_I, [ctypes.POINTER(kvsel_problem), _I, _P, ctypes.c_int64, _P, _P,
                                   _P, _P, _P, _P, _P, _P]),
    "kvsel_score_topk": (_I, [ctypes.POINTER(kvsel_problem), _P, _P, _P, _P, ctypes.c_float,
                              ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "kvsel_append_score_topk": (_I, [ctypes.POINTER(kvsel_problem), ctypes.POINTER(kvsel_append_in),
                                     _P, _P, _P, ctypes.c_float, ctypes.c_float, _P, _P, _P, _P, _P,
                                     _P, _P, _P, ctypes.c_size_t, _P]),
    "kvsel_score_topk_window": (_I, [ctypes.POINTER(kvsel_problem), ctypes.POINTER(kvsel_window),
                                     ctypes.POINTER(kvsel_append_in), _P, _P, _P, _P, ctypes.c_float,
                                     ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _P,
                                     ctypes.c_size_t, _P]),
    "kvsel_score_topk_noalloc": (_I, [ctypes.POINTER(kvsel_problem), _P, _P, _P, _P, ctypes.c_float,
                                      ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _P]),
    "kvsel_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "kvsel_set_score_path": (_I, [_I]),
    "kvsel_score_path_for": (_I, [ctypes.POINTER(kvsel_problem), _I, ctypes.POINTER(ctypes.c_int32)]),
    "kvsel_merge_spans": (_I, [ctypes.POINTER(kvsel_problem), _P, _P, _P, _P, _P, _P]),
    "kvsel_select_scores": (_I, [ctypes.POINTER(kvsel_problem), _P, _P, _P, ctypes.c_float,
                                 ctypes.c_float, _P, _P, _P, _P, _P, _P, _P]),
    "kvsel_sparse_decode": (_I, [ctypes.POINTER(kvsel_problem), _P, ctypes.POINTER(kvsel_kv_src), _P,
                                 _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P,
                                 ctypes.c_size_t, _P]),
    "kvsel_fetch_spans": (_I, [ctypes.POINTER(kvsel_problem), ctypes.POINTER(kvsel_kv_src), _P, _P, _P,
                               _P, _P, _P]),
    "kvsel_cache_reset": (_I, [ctypes.POINTER(kvsel_problem), ctypes.POINTER(kvsel_block_cache), _P]),
    "kvsel_cache_fetch": (_I, [ctypes.POINTER(kvsel_problem), ctypes.POINTER(kvsel_block_cache), _P,
                               ctypes.c_int32, _P, _P, _P, ctypes.c_int32, _P, ctypes.c_int32, _P,
                               ctypes.c_size_t, _P]),
    "kvsel_cache_prefetch": (_I, [ctypes.POINTER(kvsel_problem), ctypes.POINTER(kvsel_block_cache), _P,
                                  ctypes.c_int32, _P, _P, _P, _P, ctypes.c_int32, _P, ctypes.c_size_t,
                                  _P]),
    "kvsel_budget": (_I, [ctypes.POINTER(kvsel_budget_in), ctypes.POINTER(kvsel_budget_out)]),
    "kvsel_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(kvsel_problem), _I]),
    "kvsel_kv_bytes_per_token": (ctypes.c_int64, [ctypes.c_int32] * 4),
    "kvsel_get_error": (_I, [_P]),
    "kvsel_selftest_wait_timeout": (_I, [_P]),
    "kvsel_selftest_divide": (_I, [_P, _P, _P, ctypes.c_int64, _P]),
    "kvsel_launch_count": (ctypes.c_uint64, []),
    "kvsel_last_error": (ctypes.c_char_p, []),
    "kvsel_version": (ctypes.c_char_p, []),
}

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                        "(nvcc, sm_103a); there is no non-CUDA fallback")
                L = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGS.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = L
    return _lib


def _check(code: int, where: str):
    if code != KVSEL_OK:
        detail = lib().kvsel_last_error().decode(errors="replace")
        raise KvselError(code, where, detail)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def problem(batch, n_qheads, n_kvheads, head_dim, block_size, max_blocks, k_max=None) -> kvsel_problem:
    return kvsel_problem(int(batch), int(n_qheads), int(n_kvheads), int(head_dim), int(block_size),
                         int(max_blocks), int(k_max if k_max is not None else max_blocks))


def _expect(t, dtype, name, cuda=True):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")


# ------------------------------------------------------------ entry points ---

def kvsel_version() -> str:
    return lib().kvsel_version().decode()


def kvsel_launch_count() -> int:
    return int(lib().kvsel_launch_count())


def kvsel_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes) -> int:
    return int(lib().kvsel_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes))


def kvsel_workspace_size(p: kvsel_problem, which: int) -> int:
    return int(lib().kvsel_workspace_size(ctypes.byref(p), which))


def kvsel_set_score_path(path: int) -> int:
    """Process-wide form of the score + Top-k calls; returns the previous one."""
    prev = lib().kvsel_set_score_path(int(path))
    if prev < 0:
        raise KvselError(KVSEL_ERR_INVALID_ARG, "kvsel_set_score_path", f"unknown path {path}")
    return prev


def kvsel_score_path_for(p: kvsel_problem, with_append: bool = False):
    """(form, CTAs per cluster) a score + Top-k call on p would take."""
    ctas = ctypes.c_int32(0)
    r = lib().kvsel_score_path_for(ctypes.byref(p), int(bool(with_append)), ctypes.byref(ctas))
    if r < 0:
        _check(-r, "kvsel_score_path_for")
    return r, int(ctas.value)


def kvsel_budget(block_size, kv_heads, head_dim, elem_bytes, hidden, n_blocks, h2d_bytes_per_s,
                 recompute_flop_per_s, kappa=2.0, keep_floor=0.0, gamma=1.0, tau_s=0.0,
                 keep_override=-1.0) -> kvsel_budget_out:
    i = kvsel_budget_in(block_size, kv_heads, head_dim, elem_bytes, hidden, n_blocks,
                        h2d_bytes_per_s, recompute_flop_per_s, kappa, keep_floor, gamma, tau_s,
                        keep_override)
    o = kvsel_budget_out()
    _check(lib().kvsel_budget(ctypes.byref(i), ctypes.byref(o)), "kvsel_budget")
    return o


def kvsel_selftest_divide(x, count, out, stream=None):
    """out = x / count as the summary kernels divide a block sum by its
    token count (fp64 x and out, int32 count, device tensors)."""
    _expect(x, torch.float64, "x")
    _expect(count, torch.int32, "count")
    _expect(out, torch.float64, "out")
    _check(lib().kvsel_selftest_divide(_ptr(x), _ptr(count), _ptr(out), x.numel(), _stream(stream)),
           "kvsel_selftest_divide")


def kvsel_selftest_wait_timeout(stream=None):
    """Enqueue the bounded-wait self-test; kvsel_get_error() then returns KVSEL_ERR_TIMEOUT."""
    _check(lib().kvsel_selftest_wait_timeout(_stream(stream)), "kvsel_selftest_wait_timeout")


def kvsel_get_error(stream=None) -> int:
    return int(lib().kvsel_get_error(_stream(stream)))


def kvsel_build_summaries(p, mode, kv_pages, block_table, seq_lens, summaries, open_acc,
                          append_pos=None, new_k=None, new_v=None, stream=None):
    for t, dt, n in ((kv_pages, torch.bfloat16, "kv_pages"),
                     (block_table, torch.int32, "block_table"), (seq_lens, torch.int32, "seq_lens"),
                     (summaries, torch.bfloat16, "summaries"), (open_acc, torch.float64, "open_acc"),
                     (append_pos, torch.int32, "append_pos"), (new_k, torch.bfloat16, "new_k"),
                     (new_v, torch.bfloat16, "new_v")):
        _expect(t, dt, n)
    _check(lib().kvsel_build_summaries(ctypes.byref(p), mode, _ptr(kv_pages),
                                       kv_pages.shape[0], _ptr(block_table), _ptr(seq_lens),
                                       _ptr(append_pos), _ptr(new_k), _ptr(new_v), _ptr(summaries),
                                       _ptr(open_acc), _stream(stream)),
           "kvsel_build_summaries")


def kvsel_score_topk(p, q, summaries, seq_lens, k_per_seq, sel_idx, n_sel, span_start, span_len,
                     n_spans, ws, gamma=2.0, tau_rel=0.0, dense_flag=None, scores_out=None,
                     stream=None):
    for t, dt, n in ((q, torch.bfloat16, "q"), (summaries, torch.bfloat16, "summaries"),
                     (seq_lens, torch.int32, "seq_lens"), (k_per_seq, torch.int32, "k_per_seq"),
                     (sel_idx, torch.int32, "sel_idx"), (n_sel, torch.int32, "n_sel"),
                     (span_start, torch.int32, "span_start"), (span_len, torch.int32, "span_len"),
                     (n_spans, torch.int32, "n_spans"), (dense_flag, torch.uint8, "dense_flag"),
                     (scores_out, torch.float32, "scores_out")):
        _expect(t, dt, n)
    _check(lib().kvsel_score_topk(ctypes.byref(p), _ptr(q), _ptr(summaries), _ptr(seq_lens),
                                  _ptr(k_per_seq), float(gamma), float(tau_rel), _ptr(sel_idx),
                                  _ptr(n_sel), _ptr(span_start), _ptr(span_len), _ptr(n_spans),
                                  _ptr(dense_flag), _ptr(scores_out), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_score_topk")


def append_in(kv_pages, block_table, append_pos, summaries, open_acc, new_k=None,
              new_v=None) -> kvsel_append_in:
    """The APPEND inputs of kvsel_append_score_topk (kept alive by the caller
    together with the tensors)."""
    for t, dt, n in ((kv_pages, torch.bfloat16, "kv_pages"), (block_table, torch.int32, "block_table"),
                     (append_pos, torch.int32, "append_pos"), (summaries, torch.bfloat16, "summaries"),
                     (open_acc, torch.float64, "open_acc"), (new_k, torch.bfloat16, "new_k"),
                     (new_v, torch.bfloat16, "new_v")):
        _expect(t, dt, n)
    a = kvsel_append_in()
    a.kv_pages, a.n_pages = _ptr(kv_pages), kv_pages.shape[0]
    a.block_table, a.append_pos = _ptr(block_table), _ptr(append_pos)
    a.new_k, a.new_v = _ptr(new_k), _ptr(new_v)
    a.summaries, a.open_acc = _ptr(summaries), _ptr(open_acc)
    return a


def kvsel_append_score_topk(p, app: kvsel_append_in, q, seq_lens, k_per_seq, sel_idx, n_sel,
                            span_start, span_len, n_spans, ws, gamma=2.0, tau_rel=0.0,
                            dense_flag=None, scores_out=None, stream=None):
    """kvsel_build_summaries(APPEND) then kvsel_score_topk, in one call."""
    for t, dt, n in ((q, torch.bfloat16, "q"), (seq_lens, torch.int32, "seq_lens"),
                     (k_per_seq, torch.int32, "k_per_seq"), (sel_idx, torch.int32, "sel_idx"),
                     (n_sel, torch.int32, "n_sel"), (span_start, torch.int32, "span_start"),
                     (span_len, torch.int32, "span_len"), (n_spans, torch.int32, "n_spans"),
                     (dense_flag, torch.uint8, "dense_flag"), (scores_out, torch.float32, "scores_out")):
        _expect(t, dt, n)
    _check(lib().kvsel_append_score_topk(ctypes.byref(p), ctypes.byref(app), _ptr(q), _ptr(seq_lens),
                                         _ptr(k_per_seq), float(gamma), float(tau_rel), _ptr(sel_idx),
                                         _ptr(n_sel), _ptr(span_start), _ptr(span_len), _ptr(n_spans),
                                         _ptr(dense_flag), _ptr(scores_out), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_append_score_topk")


def kvsel_score_topk_window(p, n_sink, n_recent, q, summaries, seq_lens, k_per_seq, sel_idx,
                            n_sel, span_start, span_len, n_spans, ws, app=None, gamma=2.0,
                            tau_rel=0.0, dense_flag=None, scores_out=None, stream=None):
    """kvsel_score_topk (or, with ``app``, kvsel_append_score_topk) with the
    first ``n_sink`` and last ``n_recent`` blocks of every sequence forced
    into the selection; ``summaries`` may be None when ``app`` is given."""
    for t, dt, n in ((q, torch.bfloat16, "q"), (summaries, torch.bfloat16, "summaries"),
                     (seq_lens, torch.int32, "seq_lens"), (k_per_seq, torch.int32, "k_per_seq"),
                     (sel_idx, torch.int32, "sel_idx"), (n_sel, torch.int32, "n_sel"),
                     (span_start, torch.int32, "span_start"), (span_len, torch.int32, "span_len"),
                     (n_spans, torch.int32, "n_spans"), (dense_flag, torch.uint8, "dense_flag"),
                     (scores_out, torch.float32, "scores_out")):
        _expect(t, dt, n)
    win = kvsel_window(int(n_sink), int(n_recent))
    _check(lib().kvsel_score_topk_window(ctypes.byref(p), ctypes.byref(win),
                                         ctypes.byref(app) if app is not None else None, _ptr(q),
                                         _ptr(summaries), _ptr(seq_lens), _ptr(k_per_seq),
                                         float(gamma), float(tau_rel), _ptr(sel_idx), _ptr(n_sel),
                                         _ptr(span_start), _ptr(span_len), _ptr(n_spans),
                                         _ptr(dense_flag), _ptr(scores_out), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_score_topk_window")


def kvsel_score_topk_noalloc(p, q, summaries, seq_lens, k_per_seq, sel_idx, n_sel, span_start,
                             span_len, n_spans, gamma=2.0, tau_rel=0.0, dense_flag=None,
                             scores_out=None, stream=None):
    """kvsel_score_topk with the library's static scratch instead of a workspace."""
    for t, dt, n in ((q, torch.bfloat16, "q"), (summaries, torch.bfloat16, "summaries"),
                     (seq_lens, torch.int32, "seq_lens"), (k_per_seq, torch.int32, "k_per_seq"),
                     (sel_idx, torch.int32, "sel_idx"), (n_sel, torch.int32, "n_sel"),
                     (span_start, torch.int32, "span_start"), (span_len, torch.int32, "span_len"),
                     (n_spans, torch.int32, "n_spans"), (dense_flag, torch.uint8, "dense_flag"),
                     (scores_out, torch.float32, "scores_out")):
        _expect(t, dt, n)
    _check(lib().kvsel_score_topk_noalloc(ctypes.byref(p), _ptr(q), _ptr(summaries), _ptr(seq_lens),
                                          _ptr(k_per_seq), float(gamma), float(tau_rel),
                                          _ptr(sel_idx), _ptr(n_sel), _ptr(span_start),
                                          _ptr(span_len), _ptr(n_spans), _ptr(dense_flag),
                                          _ptr(scores_out), _stream(stream)),
           "kvsel_score_topk_noalloc")


def block_cache(slots, pool, page_of, block_in, last_use) -> kvsel_block_cache:
    """The cache descriptor (the tensors stay owned by the caller)."""
    for t, dt, n in ((pool, torch.bfloat16, "pool"), (page_of, torch.int32, "page_of"),
                     (block_in, torch.int32, "block_in"), (last_use, torch.int32, "last_use")):
        _expect(t, dt, n)
    return kvsel_block_cache(int(slots), _ptr(pool), _ptr(page_of), _ptr(block_in), _ptr(last_use))


def kvsel_cache_reset(p, cache: kvsel_block_cache, stream=None):
    _check(lib().kvsel_cache_reset(ctypes.byref(p), ctypes.byref(cache), _stream(stream)),
           "kvsel_cache_reset")


def kvsel_cache_fetch(p, cache: kvsel_block_cache, host_kv, host_blocks, seq_lens, sel_idx, n_sel,
                      step, ws, n_fetched=None, fetch_ctas=0, stream=None):
    """Serve a step's selection from the block cache, copying the misses (and
    the refreshed last block) from the pinned host tier."""
    if host_kv.is_cuda or not host_kv.is_pinned():
        raise TypeError("host_kv must be a pinned host tensor")
    for t, dt, n in ((seq_lens, torch.int32, "seq_lens"), (sel_idx, torch.int32, "sel_idx"),
                     (n_sel, torch.int32, "n_sel"), (n_fetched, torch.int32, "n_fetched")):
        _expect(t, dt, n)
    _check(lib().kvsel_cache_fetch(ctypes.byref(p), ctypes.byref(cache), _ptr(host_kv), int(host_blocks),
                                   _ptr(seq_lens), _ptr(sel_idx), _ptr(n_sel), int(step),
                                   _ptr(n_fetched), int(fetch_ctas), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_cache_fetch")


def kvsel_cache_prefetch(p, cache: kvsel_block_cache, host_kv, host_blocks, seq_lens, pred_idx, n_pred,
                         ws, n_fetched=None, fetch_ctas=0, stream=None):
    """Load a predicted block list into the block cache ahead of the
    selection that may ask for it."""
    if host_kv.is_cuda or not host_kv.is_pinned():
        raise TypeError("host_kv must be a pinned host tensor")
    for t, dt, n in ((seq_lens, torch.int32, "seq_lens"), (pred_idx, torch.int32, "pred_idx"),
                     (n_pred, torch.int32, "n_pred"), (n_fetched, torch.int32, "n_fetched")):
        _expect(t, dt, n)
    _check(lib().kvsel_cache_prefetch(ctypes.byref(p), ctypes.byref(cache), _ptr(host_kv),
                                      int(host_blocks), _ptr(seq_lens), _ptr(pred_idx), _ptr(n_pred),
                                      _ptr(n_fetched), int(fetch_ctas), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_cache_prefetch")


def kvsel_select_scores(p, scores, seq_lens, k_per_seq, sel_idx, n_sel, span_start, span_len, n_spans,
                        gamma=2.0, tau_rel=0.0, dense_flag=None, stream=None):
    for t, dt, n in ((scores, torch.float32, "scores"), (seq_lens, torch.int32, "seq_lens"),
                     (k_per_seq, torch.int32, "k_per_seq"), (sel_idx, torch.int32, "sel_idx"),
                     (n_sel, torch.int32, "n_sel"), (span_start, torch.int32, "span_start"),
                     (span_len, torch.int32, "span_len"), (n_spans, torch.int32, "n_spans"),
                     (dense_flag, torch.uint8, "dense_flag")):
        _expect(t, dt, n)
    _check(lib().kvsel_select_scores(ctypes.byref(p), _ptr(scores), _ptr(seq_lens), _ptr(k_per_seq),
                                     float(gamma), float(tau_rel), _ptr(sel_idx), _ptr(n_sel),
                                     _ptr(span_start), _ptr(span_len), _ptr(n_spans), _ptr(dense_flag),
                                     _stream(stream)),
           "kvsel_select_scores")


def kvsel_merge_spans(p, sel_idx, n_sel, span_start, span_len, n_spans, stream=None):
    for t, n in ((sel_idx, "sel_idx"), (n_sel, "n_sel"), (span_start, "span_start"),
                 (span_len, "span_len"), (n_spans, "n_spans")):
        _expect(t, torch.int32, n)
    _check(lib().kvsel_merge_spans(ctypes.byref(p), _ptr(sel_idx), _ptr(n_sel), _ptr(span_start),
                                   _ptr(span_len), _ptr(n_spans), _stream(stream)),
           "kvsel_merge_spans")


def kv_paged(kv_pages, block_table) -> kvsel_kv_src:
    _expect(kv_pages, torch.bfloat16, "kv_pages")
    _expect(block_table, torch.int32, "block_table")
    s = kvsel_kv_src()
    s.kind = KVSEL_KV_PAGED
    s.kv_pages, s.block_table = _ptr(kv_pages), _ptr(block_table)
    s.n_pages = kv_pages.shape[0]
    return s


def kv_staged(staging, slots) -> kvsel_kv_src:
    _expect(staging, torch.bfloat16, "staging")
    s = kvsel_kv_src()
    s.kind = KVSEL_KV_STAGED
    s.staging, s.staging_slots = _ptr(staging), int(slots)
    return s


def kv_host(host_kv, host_blocks, staging, slots, fetch_ctas=0) -> kvsel_kv_src:
    _expect(host_kv, torch.bfloat16, "host_kv", cuda=False)
    _expect(staging, torch.bfloat16, "staging")
    if not host_kv.is_pinned():
        raise ValueError("host_kv must be pinned host memory")
    s = kvsel_kv_src()
    s.kind = KVSEL_KV_HOST
    s.host_kv, s.host_blocks = _ptr(host_kv), int(host_blocks)
    s.staging, s.staging_slots, s.fetch_ctas = _ptr(staging), int(slots), int(fetch_ctas)
    return s


def kv_host_direct(host_kv, host_blocks) -> kvsel_kv_src:
    """The host tier read by the attention kernel itself (no staging)."""
    if host_kv.is_cuda or not host_kv.is_pinned():
        raise TypeError("host_kv must be a pinned host tensor")
    _expect(host_kv, torch.bfloat16, "host_kv", cuda=False)
    s = kvsel_kv_src()
    s.kind = KVSEL_KV_HOST_DIRECT
    s.host_kv, s.host_blocks = _ptr(host_kv), int(host_blocks)
    return s


def kvsel_sparse_decode(p, q, kv: kvsel_kv_src, seq_lens, sel_idx, n_sel, out, lse, ws,
                        softmax_scale, dense_flag=None, span_start=None, span_len=None,
                        n_spans=None, out_bf16=None, stream=None):
    for t, dt, n in ((q, torch.bfloat16, "q"), (seq_lens, torch.int32, "seq_lens"),
                     (sel_idx, torch.int32, "sel_idx"), (n_sel, torch.int32, "n_sel"),
                     (out, torch.float32, "out"), (lse, torch.float32, "lse"),
                     (dense_flag, torch.uint8, "dense_flag"), (out_bf16, torch.bfloat16, "out_bf16")):
        _expect(t, dt, n)
    _check(lib().kvsel_sparse_decode(ctypes.byref(p), _ptr(q), ctypes.byref(kv), _ptr(seq_lens),
                                     _ptr(sel_idx), _ptr(n_sel), _ptr(span_start), _ptr(span_len),
                                     _ptr(n_spans), _ptr(dense_flag), float(softmax_scale),
                                     _ptr(out), _ptr(out_bf16), _ptr(lse), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_sparse_decode")


def kvsel_fetch_spans(p, kv: kvsel_kv_src, seq_lens, span_start, span_len, n_spans,
                      dense_flag=None, stream=None):
    _check(lib().kvsel_fetch_spans(ctypes.byref(p), ctypes.byref(kv), _ptr(seq_lens),
                                   _ptr(span_start), _ptr(span_len), _ptr(n_spans),
                                   _ptr(dense_flag), _stream(stream)),
           "kvsel_fetch_spans")
