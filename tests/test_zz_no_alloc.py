"""kvsel_score_topk_noalloc: the score + Top-k entry point for callers that
cannot allocate device memory (a host framework that owns the device-memory
budget, or a path where cudaMalloc's implicit synchronisation is not
acceptable). Its scratch is the library's static device array instead of a
caller workspace.

Called through the C ABI (ctypes, no torch allocation inside the call) and
compared with kvsel_score_topk on the same inputs, on two calls in a row:
indices, spans and flags bit for bit, scores within the tolerance the parity
tests use. Without a score output the two-grid form keeps its score rows in
the static array itself, so those calls are checked too, the second one over
the first one's leftovers. This file is collected last, so a failure here
stops a run only after every other test has run; it also passes on its own in
a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from workloads import C3
from workloads.generate import generate_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from query_aware_sparse_block_gb300.build import build_library
    build_library()
    from query_aware_sparse_block_gb300 import kvsel
    kvsel.lib()
    torch.cuda.set_device(0)
    return kvsel


def _outputs(dec, scores):
    n = dec.n_sel.cpu().numpy().copy()
    ns = dec.n_spans.cpu().numpy().copy()
    return dict(n_sel=n, n_spans=ns, sel=[dec.sel_idx[b, : n[b]].cpu().numpy().copy() for b in range(len(n))],
                st=[dec.span_start[b, : ns[b]].cpu().numpy().copy() for b in range(len(ns))],
                ln=[dec.span_len[b, : ns[b]].cpu().numpy().copy() for b in range(len(ns))],
                dense=dec.dense_flag.cpu().numpy().copy(), scores=scores.cpu().numpy().copy())


def _same(a, b, N):
    assert np.array_equal(a["n_sel"], b["n_sel"]) and np.array_equal(a["n_spans"], b["n_spans"])
    assert np.array_equal(a["dense"], b["dense"])
    for x, y in zip(a["sel"], b["sel"]):
        assert np.array_equal(x, y)
    for x, y in zip(a["st"], b["st"]):
        assert np.array_equal(x, y)
    for x, y in zip(a["ln"], b["ln"]):
        assert np.array_equal(x, y)
    for r in range(len(N)):
        if N[r] == 0:
            continue
        sa, sb = a["scores"][r, : N[r]], b["scores"][r, : N[r]]
        assert np.abs(sa - sb).max() <= 1e-5 * max(1.0, np.abs(sa).max())


def test_noalloc_matches_workspace_entry_point_on_two_calls(K):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    w = C3.scaled(batch=5, seq_len=3000, drift_amp=0.0, layers=1)
    lens = [3000, 1, 2047, 0, 2999]
    x = {k: (v.to("cuda:0") if torch.is_tensor(v) else v)
         for k, v in generate_layer(w, 0, seq_lens=lens).items()}
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, x["max_blocks"],
                        k_max=40, device="cuda:0")
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.copy_(torch.tensor([12, 5, 40, 7, 33], dtype=torch.int32))
    N = [(t + w.block_size - 1) // w.block_size for t in lens]
    scores = torch.zeros((w.batch, x["max_blocks"]), device="cuda:0")
    assert K.kvsel_get_error() == 0
    dec.select(x["q"], summ, x["seq_lens"], gamma=0.5, tau_rel=0.25, scores_out=scores)
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == 0
    want = _outputs(dec, scores)

    L = K.lib()
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        for t in (dec.sel_idx, dec.n_sel, dec.span_start, dec.span_len, dec.n_spans, dec.dense_flag,
                  scores):
            t.fill_(-1 if t.dtype != torch.uint8 else 7)
        torch.cuda.synchronize()
        rc = L.kvsel_score_topk_noalloc(ctypes.byref(dec.p), vp(x["q"].data_ptr()), vp(summ.data_ptr()),
                                        vp(x["seq_lens"].data_ptr()), vp(dec.k_per_seq.data_ptr()),
                                        ctypes.c_float(0.5), ctypes.c_float(0.25),
                                        vp(dec.sel_idx.data_ptr()), vp(dec.n_sel.data_ptr()),
                                        vp(dec.span_start.data_ptr()), vp(dec.span_len.data_ptr()),
                                        vp(dec.n_spans.data_ptr()), vp(dec.dense_flag.data_ptr()),
                                        vp(scores.data_ptr()), stream)
        assert rc == 0, L.kvsel_last_error()
        torch.cuda.synchronize()
        assert K.kvsel_get_error() == 0
        _same(_outputs(dec, scores), want, N)


def test_noalloc_rejects_problems_larger_than_its_scratch(K):
    L = K.lib()
    cap = int(L.kvsel_noalloc_scratch_bytes())
    p = K.problem(4096, 32, 8, 128, 32, 16384, 128)   # needs 4096 * 16384 * 4 bytes of scores
    assert K.kvsel_workspace_size(p, K.KVSEL_WS_SCORE_TOPK) > cap
    rc = L.kvsel_score_topk_noalloc(ctypes.byref(p), None, None, None, None, ctypes.c_float(1.0),
                                    ctypes.c_float(0.0), None, None, None, None, None, None, None, None)
    assert rc == K.KVSEL_ERR_WORKSPACE
    assert b"scratch" in L.kvsel_last_error()


@pytest.mark.parametrize("path", ["two_grid", "cluster"])
def test_noalloc_scores_in_the_static_array_over_two_calls(K, path):
    """scores_out = NULL: under the two-grid form the score rows live in the
    static array. Two problems in a row with different lengths and k; the
    second call runs over the score rows the first one left behind. Every
    output equals that of the workspace entry point under the same form."""
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    w = C3.scaled(batch=4, seq_len=4096, drift_amp=0.0, layers=1)
    form = K.KVSEL_SCORE_PATH_TWO_GRID if path == "two_grid" else K.KVSEL_SCORE_PATH_CLUSTER
    L = K.lib()
    vp = ctypes.c_void_p
    runs = [([4096, 33, 4000, 1000], [40, 2, 17, 9]), ([4095, 4096, 0, 640], [3, 40, 5, 20])]
    prev = K.kvsel_set_score_path(form)
    try:
        for lens, ks in runs:
            x = {k: (v.to("cuda:0") if torch.is_tensor(v) else v)
                 for k, v in generate_layer(w, 0, seq_lens=lens).items()}
            dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size,
                                x["max_blocks"], k_max=40, device="cuda:0")
            if form == K.KVSEL_SCORE_PATH_CLUSTER:
                assert K.kvsel_score_path_for(dec.p)[0] == form
            summ, acc = dec.new_summaries()
            dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
            dec.k_per_seq.copy_(torch.tensor(ks, dtype=torch.int32))
            N = [(t + w.block_size - 1) // w.block_size for t in lens]
            dec.select(x["q"], summ, x["seq_lens"], gamma=0.6, tau_rel=0.5)
            torch.cuda.synchronize()
            assert K.kvsel_get_error() == 0
            none = torch.zeros((w.batch, x["max_blocks"]), device="cuda:0")
            want = _outputs(dec, none)
            for t in (dec.sel_idx, dec.n_sel, dec.span_start, dec.span_len, dec.n_spans, dec.dense_flag):
                t.fill_(-1 if t.dtype != torch.uint8 else 7)
            torch.cuda.synchronize()
            stream = vp(torch.cuda.current_stream().cuda_stream)
            rc = L.kvsel_score_topk_noalloc(ctypes.byref(dec.p), vp(x["q"].data_ptr()), vp(summ.data_ptr()),
                                            vp(x["seq_lens"].data_ptr()), vp(dec.k_per_seq.data_ptr()),
                                            ctypes.c_float(0.6), ctypes.c_float(0.5),
                                            vp(dec.sel_idx.data_ptr()), vp(dec.n_sel.data_ptr()),
                                            vp(dec.span_start.data_ptr()), vp(dec.span_len.data_ptr()),
                                            vp(dec.n_spans.data_ptr()), vp(dec.dense_flag.data_ptr()),
                                            None, stream)
            assert rc == 0, L.kvsel_last_error()
            torch.cuda.synchronize()
            assert K.kvsel_get_error() == 0
            _same(_outputs(dec, none), want, N)
    finally:
        K.kvsel_set_score_path(prev)
