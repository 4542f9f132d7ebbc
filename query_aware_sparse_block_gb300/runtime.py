"""Buffer ownership around the C ABI: one object per problem shape holding the
selection outputs, the workspaces and the attention outputs as torch device
tensors, with one method per library call. No arithmetic of the method runs
here; every step is a call into libkvsel.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import kvsel as K


class SparseDecoder:
    """Per-shape state for query-aware block selection + sparse decode."""

    def __init__(self, batch, n_qheads, n_kvheads, head_dim, block_size, max_blocks, k_max=None,
                 device="cuda"):
        self.p = K.problem(batch, n_qheads, n_kvheads, head_dim, block_size, max_blocks, k_max)
        self.device = torch.device(device)
        b = batch
        km = self.p.k_max
        i32 = dict(dtype=torch.int32, device=self.device)
        self.sel_idx = torch.zeros((b, km), **i32)
        self.n_sel = torch.zeros((b,), **i32)
        self.span_start = torch.zeros((b, km), **i32)
        self.span_len = torch.zeros((b, km), **i32)
        self.n_spans = torch.zeros((b,), **i32)
        self.dense_flag = torch.zeros((b,), dtype=torch.uint8, device=self.device)
        self.k_per_seq = torch.zeros((b,), **i32)
        ws1 = K.kvsel_workspace_size(self.p, K.KVSEL_WS_SCORE_TOPK)
        ws2 = K.kvsel_workspace_size(self.p, K.KVSEL_WS_SPARSE_DECODE)
        if ws1 == 0 or ws2 == 0:
            raise K.KvselError(K.KVSEL_ERR_UNSUPPORTED, "SparseDecoder",
                               K.lib().kvsel_last_error().decode())
        # no workspace needs initial contents; zero-filled only for tidiness
        self.ws_score = torch.zeros((ws1,), dtype=torch.uint8, device=self.device)
        self.ws_decode = torch.zeros((ws2,), dtype=torch.uint8, device=self.device)
        self.out = torch.zeros((b, n_qheads, head_dim), dtype=torch.float32, device=self.device)
        self.lse = torch.zeros((b, n_qheads), dtype=torch.float32, device=self.device)
        # the kernels take fp32; keep the exact value they see
        self.scale = ctypes.c_float(1.0 / math.sqrt(head_dim)).value

    def new_summaries(self):
        p = self.p
        return (torch.zeros((p.batch, p.max_blocks, p.n_kvheads, p.head_dim), dtype=torch.bfloat16,
                            device=self.device),
                torch.zeros((p.batch, p.n_kvheads, p.head_dim), dtype=torch.float64, device=self.device))

    def build_summaries(self, kv_pages, block_table, seq_lens, summaries, open_acc, stream=None):
        K.kvsel_build_summaries(self.p, K.KVSEL_SUMMARY_FULL, kv_pages, block_table, seq_lens,
                                summaries, open_acc, stream=stream)

    def append(self, kv_pages, block_table, append_pos, summaries, open_acc, new_k=None,
               new_v=None, stream=None):
        K.kvsel_build_summaries(self.p, K.KVSEL_SUMMARY_APPEND, kv_pages, block_table, None,
                                summaries, open_acc, append_pos=append_pos, new_k=new_k, new_v=new_v,
                                stream=stream)

    def select(self, q, summaries, seq_lens, k_per_seq=None, gamma=2.0, tau_rel=0.0,
               scores_out=None, stream=None):
        kp = self.k_per_seq if k_per_seq is None else k_per_seq
        K.kvsel_score_topk(self.p, q, summaries, seq_lens, kp, self.sel_idx, self.n_sel,
                           self.span_start, self.span_len, self.n_spans, self.ws_score,
                           gamma=gamma, tau_rel=tau_rel, dense_flag=self.dense_flag,
                           scores_out=scores_out, stream=stream)

    def append_select(self, kv_pages, block_table, append_pos, q, summaries, open_acc, seq_lens,
                      new_k=None, new_v=None, k_per_seq=None, gamma=2.0, tau_rel=0.0,
                      scores_out=None, stream=None):
        """append() then select() as one call (kvsel_append_score_topk)."""
        kp = self.k_per_seq if k_per_seq is None else k_per_seq
        app = K.append_in(kv_pages, block_table, append_pos, summaries, open_acc, new_k, new_v)
        K.kvsel_append_score_topk(self.p, app, q, seq_lens, kp, self.sel_idx, self.n_sel,
                                  self.span_start, self.span_len, self.n_spans, self.ws_score,
                                  gamma=gamma, tau_rel=tau_rel, dense_flag=self.dense_flag,
                                  scores_out=scores_out, stream=stream)

    def select_window(self, q, summaries, seq_lens, n_sink, n_recent, k_per_seq=None, gamma=2.0,
                      tau_rel=0.0, scores_out=None, app=None, stream=None):
        """select() with the first n_sink and last n_recent blocks forced in
        (kvsel_score_topk_window); ``app`` (kvsel.append_in) folds the
        token's append into the call as append_select() does."""
        kp = self.k_per_seq if k_per_seq is None else k_per_seq
        K.kvsel_score_topk_window(self.p, n_sink, n_recent, q, summaries, seq_lens, kp, self.sel_idx,
                                  self.n_sel, self.span_start, self.span_len, self.n_spans,
                                  self.ws_score, app=app, gamma=gamma, tau_rel=tau_rel,
                                  dense_flag=self.dense_flag, scores_out=scores_out, stream=stream)

    def attend(self, q, kv, seq_lens, use_dense_flag=True, out=None, lse=None, out_bf16=None,
               stream=None):
        K.kvsel_sparse_decode(self.p, q, kv, seq_lens, self.sel_idx, self.n_sel,
                              self.out if out is None else out, self.lse if lse is None else lse,
                              self.ws_decode, self.scale,
                              dense_flag=self.dense_flag if use_dense_flag else None,
                              span_start=self.span_start, span_len=self.span_len,
                              n_spans=self.n_spans, out_bf16=out_bf16, stream=stream)


class BoundLayer:
    """Pre-marshalled C-ABI calls for one layer's fixed buffers.

    A decode loop calls the same three entry points with the same buffers on
    every step; only the step's position / length arrays and the stream
    change. Converting every argument once keeps the host-side cost of a call
    to a few microseconds, so the host enqueues ahead of the GPU.
    """

    def __init__(self, dec: SparseDecoder, q, kv_pages, block_table, summaries, open_acc,
                 out, lse, kv=None, gamma=2.0, tau_rel=0.0, new_k=None, new_v=None, window=None):
        """``window`` = (n_sink, n_recent) makes append_select() force those
        blocks into the selection (kvsel_score_topk_window)."""
        L = K.lib()
        vp = ctypes.c_void_p
        self._fa, self._fs, self._fd = L.kvsel_build_summaries, L.kvsel_score_topk, L.kvsel_sparse_decode
        self._fas = L.kvsel_append_score_topk
        self._fw = L.kvsel_score_topk_window
        self._win = K.kvsel_window(*window) if window is not None else None
        self._win_ref = ctypes.byref(self._win) if window is not None else None
        self.dec = dec
        self.p = ctypes.byref(dec.p)
        self.kv = kv if kv is not None else K.kv_paged(kv_pages, block_table)
        self.kv_ref = ctypes.byref(self.kv)
        self.kv_pages = vp(kv_pages.data_ptr())
        self.n_pages = int(kv_pages.shape[0])
        self.block_table = vp(block_table.data_ptr())
        self.q = vp(q.data_ptr())
        self.summ, self.acc = vp(summaries.data_ptr()), vp(open_acc.data_ptr())
        self.new_k = vp(new_k.data_ptr()) if new_k is not None else None
        self.new_v = vp(new_v.data_ptr()) if new_v is not None else None
        self.out, self.lse = vp(out.data_ptr()), vp(lse.data_ptr())
        self.gamma, self.tau = ctypes.c_float(gamma), ctypes.c_float(tau_rel)
        d = dec
        self.sel = (vp(d.sel_idx.data_ptr()), vp(d.n_sel.data_ptr()), vp(d.span_start.data_ptr()),
                    vp(d.span_len.data_ptr()), vp(d.n_spans.data_ptr()), vp(d.dense_flag.data_ptr()))
        self.kps = vp(d.k_per_seq.data_ptr())
        self.ws1, self.ws1n = vp(d.ws_score.data_ptr()), ctypes.c_size_t(d.ws_score.numel())
        self.ws2, self.ws2n = vp(d.ws_decode.data_ptr()), ctypes.c_size_t(d.ws_decode.numel())
        self.scale = ctypes.c_float(d.scale)
        self._app = K.kvsel_append_in()
        self._app.kv_pages, self._app.n_pages = self.kv_pages.value, self.n_pages
        self._app.block_table = self.block_table.value
        self._app.summaries, self._app.open_acc = self.summ.value, self.acc.value
        self._app_ref = ctypes.byref(self._app)

    def append(self, append_pos_ptr, stream_ptr, new_k_ptr=None, new_v_ptr=None):
        nk = new_k_ptr if new_k_ptr is not None else self.new_k
        nv = new_v_ptr if new_v_ptr is not None else self.new_v
        rc = self._fa(self.p, K.KVSEL_SUMMARY_APPEND, self.kv_pages, self.n_pages,
                      self.block_table, None, append_pos_ptr, nk, nv, self.summ, self.acc, stream_ptr)
        if rc:
            K._check(rc, "kvsel_build_summaries")

    def append_select(self, append_pos_ptr, seq_lens_ptr, stream_ptr, new_k_ptr=None,
                      new_v_ptr=None, q_ptr=None):
        """append() and select() folded into one call (kvsel_append_score_topk)."""
        app = self._app
        app.append_pos = append_pos_ptr.value if isinstance(append_pos_ptr, ctypes.c_void_p) else append_pos_ptr
        nk = new_k_ptr if new_k_ptr is not None else self.new_k
        nv = new_v_ptr if new_v_ptr is not None else self.new_v
        app.new_k = nk.value if isinstance(nk, ctypes.c_void_p) else nk
        app.new_v = nv.value if isinstance(nv, ctypes.c_void_p) else nv
        s = self.sel
        qp = q_ptr if q_ptr is not None else self.q
        if self._win is not None:
            rc = self._fw(self.p, self._win_ref, self._app_ref, qp, None, seq_lens_ptr, self.kps,
                          self.gamma, self.tau, s[0], s[1], s[2], s[3], s[4], s[5], None,
                          self.ws1, self.ws1n, stream_ptr)
            if rc:
                K._check(rc, "kvsel_score_topk_window")
            return
        rc = self._fas(self.p, self._app_ref, qp, seq_lens_ptr,
                       self.kps, self.gamma, self.tau, s[0], s[1], s[2], s[3], s[4], s[5], None,
                       self.ws1, self.ws1n, stream_ptr)
        if rc:
            K._check(rc, "kvsel_append_score_topk")

    def select(self, seq_lens_ptr, stream_ptr, q_ptr=None):
        s = self.sel
        rc = self._fs(self.p, q_ptr if q_ptr is not None else self.q, self.summ, seq_lens_ptr,
                      self.kps, self.gamma, self.tau, s[0], s[1], s[2], s[3], s[4], s[5], None,
                      self.ws1, self.ws1n, stream_ptr)
        if rc:
            K._check(rc, "kvsel_score_topk")

    def attend(self, seq_lens_ptr, stream_ptr, q_ptr=None, out_ptr=None):
        s = self.sel
        rc = self._fd(self.p, q_ptr if q_ptr is not None else self.q, self.kv_ref, seq_lens_ptr,
                      s[0], s[1], s[2], s[3], s[4], s[5], self.scale,
                      out_ptr if out_ptr is not None else self.out, None, self.lse,
                      self.ws2, self.ws2n, stream_ptr)
        if rc:
            K._check(rc, "kvsel_sparse_decode")


class HostBlockCache:
    """Device buffers of a GPU-resident cache of host-tier blocks
    (kvsel_cache_fetch): ``slots`` pool pages per sequence, the block/slot
    maps and a step counter. After fetch(), ``kv`` is the paged view of the
    pool that kvsel_sparse_decode reads (dense flag off)."""

    def __init__(self, dec: SparseDecoder, slots, page_shape):
        p = dec.p
        self.p, self.slots, self.device = p, int(slots), dec.device
        i32 = dict(dtype=torch.int32, device=self.device)
        self.pool = torch.empty((p.batch * self.slots,) + tuple(page_shape), dtype=torch.bfloat16,
                                device=self.device)
        self.page_of = torch.empty((p.batch, p.max_blocks), **i32)
        self.block_in = torch.empty((p.batch, self.slots), **i32)
        self.last_use = torch.empty((p.batch, self.slots), **i32)
        self.n_fetched = torch.zeros((p.batch,), **i32)
        self.n_prefetched = torch.zeros((p.batch,), **i32)
        self.ws = torch.zeros((K.kvsel_workspace_size(p, K.KVSEL_WS_CACHE_FETCH),), dtype=torch.uint8,
                              device=self.device)
        self.desc = K.block_cache(self.slots, self.pool, self.page_of, self.block_in, self.last_use)
        self.kv = K.kv_paged(self.pool, self.page_of)
        self.step = 0
        self.reset()

    def reset(self, stream=None):
        K.kvsel_cache_reset(self.p, self.desc, stream=stream)
        self.step = 0

    def fetch(self, host_kv, host_blocks, seq_lens, sel_idx, n_sel, fetch_ctas=0, stream=None):
        K.kvsel_cache_fetch(self.p, self.desc, host_kv, host_blocks, seq_lens, sel_idx, n_sel,
                            self.step, self.ws, n_fetched=self.n_fetched, fetch_ctas=fetch_ctas,
                            stream=stream)
        self.step += 1

    def prefetch(self, host_kv, host_blocks, seq_lens, pred_idx, n_pred, fetch_ctas=0, stream=None):
        """Load a predicted block list (e.g. BlockPredictor.pred_idx) ahead
        of the next fetch(); order that fetch after this call."""
        K.kvsel_cache_prefetch(self.p, self.desc, host_kv, host_blocks, seq_lens, pred_idx, n_pred,
                               self.ws, n_fetched=self.n_prefetched, fetch_ctas=fetch_ctas,
                               stream=stream)


class BlockPredictor:
    """The blocks a layer is expected to select at its next step, with no
    trained predictor: the k_pred highest-scoring blocks of its score rows
    from the current step (kvsel_select_scores on the rows a score call wrote
    to scores_out). Selections of consecutive steps overlap ("KV cache
    offloading", section "NOSA"), and the blocks that enter the next
    selection come mostly from just below this step's k-th score, so a list
    wider than k covers part of the next step's misses."""

    def __init__(self, dec: SparseDecoder, k_pred):
        p = dec.p
        if not 0 < int(k_pred) <= p.k_max:
            raise ValueError("k_pred must be in [1, k_max]")
        self.p, self.device = p, dec.device
        i32 = dict(dtype=torch.int32, device=self.device)
        self.k_pred = torch.full((p.batch,), int(k_pred), **i32)
        self.pred_idx = torch.zeros((p.batch, p.k_max), **i32)
        self.n_pred = torch.zeros((p.batch,), **i32)
        self.span_start = torch.zeros((p.batch, p.k_max), **i32)
        self.span_len = torch.zeros((p.batch, p.k_max), **i32)
        self.n_spans = torch.zeros((p.batch,), **i32)

    def from_scores(self, scores, seq_lens, stream=None):
        K.kvsel_select_scores(self.p, scores, seq_lens, self.k_pred, self.pred_idx, self.n_pred,
                              self.span_start, self.span_len, self.n_spans, stream=stream)
