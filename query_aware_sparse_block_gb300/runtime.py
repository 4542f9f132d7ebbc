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
        # workspaces start zero-filled; the kernels leave them zero-filled
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

    def build_summaries(self, k_pages, block_table, seq_lens, summaries, open_acc, stream=None):
        K.kvsel_build_summaries(self.p, K.KVSEL_SUMMARY_FULL, k_pages, None, block_table, seq_lens,
                                summaries, open_acc, stream=stream)

    def append(self, k_pages, v_pages, block_table, append_pos, summaries, open_acc, new_k=None,
               new_v=None, stream=None):
        K.kvsel_build_summaries(self.p, K.KVSEL_SUMMARY_APPEND, k_pages, v_pages, block_table, None,
                                summaries, open_acc, append_pos=append_pos, new_k=new_k, new_v=new_v,
                                stream=stream)

    def select(self, q, summaries, seq_lens, k_per_seq=None, gamma=2.0, tau_rel=0.0,
               scores_out=None, stream=None):
        kp = self.k_per_seq if k_per_seq is None else k_per_seq
        K.kvsel_score_topk(self.p, q, summaries, seq_lens, kp, self.sel_idx, self.n_sel,
                           self.span_start, self.span_len, self.n_spans, self.ws_score,
                           gamma=gamma, tau_rel=tau_rel, dense_flag=self.dense_flag,
                           scores_out=scores_out, stream=stream)

    def attend(self, q, kv, seq_lens, use_dense_flag=True, out=None, lse=None, out_bf16=None,
               stream=None):
        K.kvsel_sparse_decode(self.p, q, kv, seq_lens, self.sel_idx, self.n_sel,
                              self.out if out is None else out, self.lse if lse is None else lse,
                              self.ws_decode, self.scale,
                              dense_flag=self.dense_flag if use_dense_flag else None,
                              span_start=self.span_start, span_len=self.span_len,
                              n_spans=self.n_spans, out_bf16=out_bf16, stream=stream)
