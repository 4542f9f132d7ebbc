"""GPU: kvsel_score_topk_window (the first n_sink and last n_recent blocks of
every sequence forced into the selection, Top-k over the blocks between)
against the fp64 oracle's window_select, element by element on small ragged
cases and on sampled sequences of the Qwen3-4B-shaped batch at full size; a
zero window against kvsel_score_topk bit for bit; the folded append against
the separate APPEND call bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as o
from tests._parity import (ATOL_MAX, ATOL_MEAN, attn_errors, seq_inputs, selection_verdict,
                           to_dev)
from workloads import C0, C2, C3
from workloads.generate import bits, generate_layer

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


@pytest.fixture(autouse=True)
def _no_device_error(K):
    K.kvsel_get_error()
    yield
    assert K.kvsel_get_error() == 0, "a kernel latched a device error"


def _decoder(w, mb, k_max=None):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    return SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, mb,
                         k_max=k_max, device="cuda:0")


def window_verdict(scores, k, n_sink, n_recent, gpu_sel):
    """The forced blocks must match exactly; the Top-k part follows the tie
    rule of the plain selection on the candidate blocks."""
    N = len(scores)
    lo = min(n_sink, N)
    hi = max(lo, N - n_recent)
    gpu_sel = np.asarray(gpu_sel, dtype=np.int64)
    forced = gpu_sel[(gpu_sel < lo) | (gpu_sel >= hi)]
    assert forced.tolist() == list(range(lo)) + list(range(hi, N))
    picks = gpu_sel[(gpu_sel >= lo) & (gpu_sel < hi)] - lo
    v = selection_verdict(scores[lo:hi], min(k, hi - lo), picks)
    if v == "exact":
        assert np.array_equal(gpu_sel, o.window_select(scores, k, n_sink, n_recent))
    return v


def check_window_sequence(dec, x, b, T, B, k, n_sink, n_recent, scale, gamma=2.0, scores_gpu=None):
    qb, kb, vb = seq_inputs(x, b, T)
    N = o.n_blocks(T, B)
    sb = o.block_summaries(kb, T, B)[0] if T > 0 else None
    scores = o.block_scores(qb, sb) if N > 0 else np.zeros(0)
    if scores_gpu is not None and N > 0:
        sg = scores_gpu[b, :N].double().cpu().numpy()
        assert np.abs(sg - scores).max() <= 1e-5 * max(1.0, np.abs(scores).max())
    n = int(dec.n_sel[b])
    gsel = dec.sel_idx[b, :n].cpu().numpy().astype(np.int64)
    verdict = window_verdict(scores, k, n_sink, n_recent, gsel)
    st, ln = o.merge_spans(gsel)
    ns = int(dec.n_spans[b])
    assert ns == len(st)
    assert np.array_equal(dec.span_start[b, :ns].cpu().numpy(), st)
    assert np.array_equal(dec.span_len[b, :ns].cpu().numpy(), ln)
    dense = N > 0 and o.dense_fallback(len(st), len(gsel), N, gamma, 0.0)
    assert bool(dec.dense_flag[b]) == dense
    blocks = np.arange(N) if dense else gsel
    ref, ref_lse = o.attend(qb, kb, vb, o.tokens_of_blocks(blocks, T, B), scale)
    emax, emean = attn_errors(dec.out[b].double().cpu().numpy(), ref)
    assert emax <= ATOL_MAX and emean <= ATOL_MEAN, (b, emax, emean)
    lse = dec.lse[b].double().cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-3 * max(1.0, np.abs(ref_lse[fin]).max())
    return verdict


SMALL = [
    # name, workload, seq_lens, k, n_sink, n_recent
    ("mha_d64_B16_sink1_recent2", C0.scaled(batch=3, seq_len=1000), [1000, 37, 513], 7, 1, 2),
    ("mha_d64_B16_recent5", C0.scaled(batch=3, seq_len=1000), [1000, 90, 1], 9, 0, 5),
    ("gqa4_d128_B32_sink3", C3.scaled(batch=3, seq_len=2000, drift_amp=0.0, layers=1), [2000, 100, 1999], 6, 3, 0),
    ("gqa4_d128_B32_sink2_recent4", C3.scaled(batch=3, seq_len=3000, drift_amp=0.0, layers=1), [3000, 150, 2500], 20, 2, 4),
    ("gqa16_d128_B64_recent8", C2.scaled(batch=2, seq_len=9000, layers=1), [9000, 4097], 5, 1, 8),
    ("k0_window_only_and_empty", C0.scaled(batch=3, seq_len=320), [320, 0, 40], 0, 1, 3),
]


@pytest.mark.parametrize("name,w,lens,k,n_sink,n_recent", SMALL, ids=[s[0] for s in SMALL])
def test_window_small_cases_elementwise(K, name, w, lens, k, n_sink, n_recent):
    x = to_dev(generate_layer(w, 0, seq_lens=lens), "cuda:0")
    mb = x["max_blocks"]
    dec = _decoder(w, mb, k_max=max(1, k + n_sink + n_recent))
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.fill_(k)
    scores = torch.full((w.batch, mb), float("nan"), device="cuda:0")
    dec.select_window(x["q"], summ, x["seq_lens"], n_sink, n_recent, scores_out=scores)
    dec.attend(x["q"], K.kv_paged(x["kv_pages"], x["block_table"]), x["seq_lens"])
    torch.cuda.synchronize()
    for b in range(w.batch):
        check_window_sequence(dec, x, b, lens[b], w.block_size, k, n_sink, n_recent, dec.scale,
                              scores_gpu=scores)


def test_zero_window_equals_plain_selection_bit_for_bit(K):
    w = C3.scaled(batch=4, seq_len=4000, drift_amp=0.0, layers=1)
    x = to_dev(generate_layer(w, 0, seq_lens=[4000, 3000, 45, 2999]), "cuda:0")
    mb = x["max_blocks"]
    da, db = _decoder(w, mb, k_max=24), _decoder(w, mb, k_max=24)
    summ, acc = da.new_summaries()
    da.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    for d in (da, db):
        d.k_per_seq.fill_(17)
    da.select(x["q"], summ, x["seq_lens"], gamma=0.5)
    db.select_window(x["q"], summ, x["seq_lens"], 0, 0, gamma=0.5)
    torch.cuda.synchronize()
    for name in ("sel_idx", "n_sel", "span_start", "span_len", "n_spans", "dense_flag"):
        assert torch.equal(getattr(da, name), getattr(db, name)), name


def test_window_with_folded_append_equals_separate_calls(K):
    w = C3.scaled(batch=3, seq_len=600, drift_amp=0.0, layers=1)
    B = w.block_size
    lens0 = [600, 431, 64]
    steps = 40
    mb = (max(lens0) + steps + B - 1) // B
    x = to_dev(generate_layer(w, 0, max_blocks=mb, seq_lens=lens0), "cuda:0")
    pa, pb = x["kv_pages"].clone(), x["kv_pages"].clone()
    da, db = _decoder(w, mb, k_max=12), _decoder(w, mb, k_max=12)
    sa, aa = da.new_summaries()
    sb, ab = db.new_summaries()
    da.build_summaries(pa, x["block_table"], x["seq_lens"], sa, aa)
    db.build_summaries(pb, x["block_table"], x["seq_lens"], sb, ab)
    for d in (da, db):
        d.k_per_seq.fill_(7)
    g = torch.Generator(device="cuda:0")
    g.manual_seed(3)
    lens = x["seq_lens"].clone()
    for step in range(steps):
        shape = (w.batch, w.n_kvheads, w.head_dim)
        nk = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
        nv = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
        q = torch.randn((w.batch, w.n_qheads, w.head_dim), generator=g, device="cuda:0").to(torch.bfloat16)
        pos = lens.clone()
        lens += 1
        app = K.append_in(pa, x["block_table"], pos, sa, aa, nk, nv)
        da.select_window(q, None, lens, 2, 3, app=app)
        db.append(pb, x["block_table"], pos, sb, ab, new_k=nk, new_v=nv)
        db.select_window(q, sb, lens, 2, 3)
        torch.cuda.synchronize()
        assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
        assert torch.equal(sa.view(torch.int16), sb.view(torch.int16))
        assert torch.equal(aa, ab)
        for name in ("sel_idx", "n_sel", "span_start", "span_len", "n_spans", "dense_flag"):
            assert torch.equal(getattr(da, name), getattr(db, name)), (step, name)
    # the final state against the oracle
    x["kv_pages"], x["seq_lens"], x["q"] = pa, lens, q
    da.attend(q, K.kv_paged(pa, x["block_table"]), lens)
    torch.cuda.synchronize()
    for b in range(w.batch):
        check_window_sequence(da, x, b, int(lens[b]), B, 7, 2, 3, da.scale)


def test_window_dense_fallback_counts_forced_blocks(K):
    # N = 10 blocks, 3 forced (1 sink, 2 recent), gamma 0.75 (exact in fp32):
    # 3 + 5 = 8 >= 7.5 goes dense, 3 + 4 = 7 < 7.5 stays sparse
    w = C0.scaled(batch=2, seq_len=160)
    x = to_dev(generate_layer(w, 0, seq_lens=[160, 159]), "cuda:0")
    dec = _decoder(w, x["max_blocks"], k_max=10)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    ks = [5, 4]
    dec.k_per_seq.copy_(torch.tensor(ks, dtype=torch.int32))
    dec.select_window(x["q"], summ, x["seq_lens"], 1, 2, gamma=0.75)
    dec.attend(x["q"], K.kv_paged(x["kv_pages"], x["block_table"]), x["seq_lens"])
    torch.cuda.synchronize()
    assert dec.dense_flag.cpu().tolist() == [1, 0]
    for b in range(2):
        check_window_sequence(dec, x, b, int(x["seq_lens"][b]), w.block_size, ks[b], 1, 2, dec.scale,
                              gamma=0.75)


def test_window_oversized_k_is_clamped_and_latched(K):
    w = C0.scaled(batch=1, seq_len=320)
    x = to_dev(generate_layer(w, 0), "cuda:0")
    dec = _decoder(w, x["max_blocks"], k_max=10)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.fill_(8)              # 8 + 5 forced > k_max
    dec.select_window(x["q"], summ, x["seq_lens"], 2, 3)
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS
    n = int(dec.n_sel[0])
    assert n == 10
    sel = dec.sel_idx[0, :n].cpu().tolist()
    N = 20
    assert sel[:2] == [0, 1] and sel[-3:] == [N - 3, N - 2, N - 1]
    qb, kb, _ = seq_inputs(x, 0, 320)
    sc = o.block_scores(qb, o.block_summaries(kb, 320, w.block_size)[0])
    window_verdict(sc, 5, 2, 3, np.array(sel))


def test_c3_full_size_window(K):
    """Qwen3-4B-shaped batch at full size (16 sequences of 32768 tokens, 1024
    blocks, Top-k 128) with one sink block and a 4-block recency window, in
    the launch configuration of the bench; sampled sequences against the
    oracle."""
    w = C3
    k = w.k_for(w.keep[0])
    x = generate_layer(w, 0, device="cuda:0", perm=True)
    mb = x["max_blocks"]
    dec = _decoder(w, mb, k_max=k + 5)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.fill_(k)
    scores = torch.full((w.batch, mb), float("nan"), device="cuda:0")
    dec.select_window(x["q"], summ, x["seq_lens"], 1, 4, scores_out=scores)
    dec.attend(x["q"], K.kv_paged(x["kv_pages"], x["block_table"]), x["seq_lens"])
    torch.cuda.synchronize()
    assert dec.n_sel.cpu().tolist() == [k + 5] * w.batch
    for b in (0, 7, 15):
        check_window_sequence(dec, x, b, w.seq_len, w.block_size, k, 1, 4, dec.scale, scores_gpu=scores)
