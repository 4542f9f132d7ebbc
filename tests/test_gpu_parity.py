"""GPU parity: every kernel through the C ABI against the fp64 oracle.

Small cases span several tiles and ragged tails and are checked element by
element; the five workload shapes run at full size in the launch
configuration the bench uses and are checked on sampled sequences.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as o
from tests._parity import (attn_errors, check_sequence, default_scale, seq_inputs, selection_verdict,
                           to_dev)
from workloads import C0, C1, C2, C3, C4, Workload
from workloads.generate import bits, generate_layer, host_tier_layout, logical_kv, natural_blocks

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


def _decoder(w, x, k_max=None):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    return SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size,
                         x["max_blocks"], k_max=k_max, device="cuda:0")


def _run(K, w, x, k, gamma=2.0, tau_rel=0.0, k_per_seq=None, use_scores=True):
    dec = _decoder(w, x)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    if k_per_seq is None:
        dec.k_per_seq.fill_(k)
    else:
        dec.k_per_seq.copy_(torch.as_tensor(k_per_seq, dtype=torch.int32))
    scores = torch.full((w.batch, x["max_blocks"]), float("nan"), device="cuda:0") if use_scores else None
    dec.select(x["q"], summ, x["seq_lens"], gamma=gamma, tau_rel=tau_rel, scores_out=scores)
    dec.attend(x["q"], K.kv_paged(x["kv_pages"], x["block_table"]), x["seq_lens"])
    torch.cuda.synchronize()
    return dec, summ, acc, scores


SMALL = [
    # name, workload, seq_lens, k
    ("c0", C0, None, 16),
    ("mha_d64_B16_ragged", C0.scaled(batch=3, seq_len=1000), [1000, 37, 513], 7),
    ("gqa4_d128_B32_ragged", C3.scaled(batch=3, seq_len=2000, drift_amp=0.0, layers=1), [2000, 1, 1999], 9),
    ("gqa16_d128_B64", C2.scaled(batch=2, seq_len=5000, layers=1), [5000, 4097], 5),
    ("gqa2_d64_B32", C0.scaled(n_qheads=8, n_kvheads=4, block_size=32, batch=2, seq_len=777), [777, 700], 6),
    ("mha_d128_B16", C1.scaled(batch=2, seq_len=900, layers=1, needles=()), [900, 899], 11),
]


@pytest.mark.parametrize("name,w,lens,k", SMALL, ids=[s[0] for s in SMALL])
def test_small_cases_elementwise(K, name, w, lens, k):
    x = to_dev(generate_layer(w, 0, seq_lens=lens), "cuda:0")
    dec, summ, acc, scores = _run(K, w, x, k)
    T = x["seq_lens"].cpu().tolist()
    for b in range(w.batch):
        check_sequence(dec, x, b, T[b], w.block_size, k, dec.scale, scores_gpu=scores,
                       summaries_gpu=summ)
        # open-block accumulator = fp64 sum of the last block
        kb = seq_inputs(x, b, T[b])[1]
        _, _, last = o.block_summaries(kb, T[b], w.block_size)
        assert np.array_equal(acc[b].cpu().numpy(), last)


def test_incremental_append_equals_rebuild_and_writes_cache(K):
    w = C3.scaled(batch=2, seq_len=200, drift_amp=0.0, layers=1)
    T0, T1 = 150, 200
    x = to_dev(generate_layer(w, 0, max_blocks=8, seq_lens=[T0, T0 - 7]), "cuda:0")
    dec = _decoder(w, x)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    g = torch.Generator(device="cuda:0")
    g.manual_seed(5)
    lens = x["seq_lens"].clone()
    for step in range(T1 - T0):
        new_k = torch.randn((w.batch, w.n_kvheads, w.head_dim), generator=g, device="cuda:0").to(torch.bfloat16)
        new_v = torch.randn((w.batch, w.n_kvheads, w.head_dim), generator=g, device="cuda:0").to(torch.bfloat16)
        pos = lens.clone()
        dec.append(x["kv_pages"], x["block_table"], pos, summ, acc, new_k=new_k, new_v=new_v)
        lens += 1
    torch.cuda.synchronize()
    x["seq_lens"] = lens
    summ2, acc2 = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], lens, summ2, acc2)
    torch.cuda.synchronize()
    for b in range(w.batch):
        T = int(lens[b])
        kb = seq_inputs(x, b, T)[1]
        sb, _, last = o.block_summaries(kb, T, w.block_size)
        N = sb.shape[0]
        assert np.array_equal(bits(summ[b, :N]), sb)
        assert np.array_equal(bits(summ2[b, :N]), sb)
        assert np.array_equal(acc[b].cpu().numpy(), last)


def test_topk_exact_ties_take_lower_index(K):
    w = C0.scaled(batch=1, seq_len=64 * 16)
    x = to_dev(generate_layer(w, 0), "cuda:0")
    # make blocks 40..63 copies of blocks 0..23 so that their scores tie exactly
    B = w.block_size
    tbl = x["block_table"][0]
    for n in range(40, 64):
        x["kv_pages"][tbl[n], :, 0] = x["kv_pages"][tbl[n - 40], :, 0]
    dec, summ, _, scores = _run(K, w, x, 20)
    sc = scores[0, :64].cpu().numpy()
    assert np.array_equal(sc[40:64], sc[0:24])
    want = o.topk_blocks(sc.astype(np.float64), 20)    # fp32 scores, exact ties
    got = dec.sel_idx[0, : int(dec.n_sel[0])].cpu().numpy()
    assert np.array_equal(got, want)


def test_merge_spans_kernel(K):
    p = K.problem(5, 8, 8, 64, 16, 64, 40)
    rng = np.random.default_rng(0)
    sel = np.zeros((5, 40), np.int32)
    nsel = np.zeros(5, np.int32)
    for b in range(5):
        k = int(rng.integers(0, 41))
        s = np.sort(rng.choice(64, size=k, replace=False))
        sel[b, :k] = s
        nsel[b] = k
    d = torch.device("cuda:0")
    ts, tn = torch.from_numpy(sel).to(d), torch.from_numpy(nsel).to(d)
    st = torch.zeros((5, 40), dtype=torch.int32, device=d)
    ln = torch.zeros_like(st)
    ns = torch.zeros(5, dtype=torch.int32, device=d)
    K.kvsel_merge_spans(p, ts, tn, st, ln, ns)
    torch.cuda.synchronize()
    for b in range(5):
        a, l = o.merge_spans(sel[b, : nsel[b]])
        n = int(ns[b])
        assert n == len(a)
        assert np.array_equal(st[b, :n].cpu().numpy(), a) and np.array_equal(ln[b, :n].cpu().numpy(), l)


@pytest.mark.parametrize("gamma,tau", [(0.0, 0.0), (0.25, 0.0), (0.3, 2.0), (1.0, 0.0)])
def test_dense_fallback_rule_and_full_attention(K, gamma, tau):
    w = C3.scaled(batch=3, seq_len=1500, drift_amp=0.0, layers=1)
    x = to_dev(generate_layer(w, 0, seq_lens=[1500, 700, 33]), "cuda:0")
    dec, summ, _, scores = _run(K, w, x, 12, gamma=gamma, tau_rel=tau)
    for b in range(w.batch):
        check_sequence(dec, x, b, int(x["seq_lens"][b]), w.block_size, 12, dec.scale, gamma=gamma,
                       tau_rel=tau)


def test_k_equal_all_blocks_is_full_attention(K):
    w = C0.scaled(batch=2, seq_len=500, n_qheads=8, n_kvheads=2)
    x = to_dev(generate_layer(w, 0, seq_lens=[500, 260]), "cuda:0")
    dec, *_ = _run(K, w, x, o.n_blocks(500, w.block_size))     # k = every block of the longest
    for b in range(2):
        T = int(x["seq_lens"][b])
        qb, kb, vb = seq_inputs(x, b, T)
        ref, ref_lse = o.attend(qb, kb, vb, np.arange(T), dec.scale)
        emax, emean = attn_errors(dec.out[b].cpu().numpy(), ref)
        assert emax <= 1e-2 and emean <= 1e-3
        assert int(dec.n_sel[b]) == o.n_blocks(T, w.block_size)


def test_empty_and_degenerate_sequences(K):
    w = C0.scaled(batch=4, seq_len=256)
    x = to_dev(generate_layer(w, 0, seq_lens=[0, 256, 1, 0]), "cuda:0")
    dec, *_ = _run(K, w, x, 4, k_per_seq=[4, 0, 4, 4])
    n_sel = dec.n_sel.cpu().tolist()
    assert n_sel == [0, 0, 1, 0]
    for b in (0, 1, 3):
        assert torch.all(dec.out[b] == 0) and torch.all(torch.isneginf(dec.lse[b]))
    check_sequence(dec, x, 2, 1, w.block_size, 4, dec.scale)


@pytest.mark.parametrize("name,w,lens,k,gamma", [
    # equal non-empty segments with empty sequences between them: the decode's
    # equal-segment split, its CTAs mapped past the empty ones
    ("equal_with_empty", C3.scaled(batch=7, seq_len=3000, layers=1),
     [3000, 0, 3000, 3000, 0, 0, 3000], 24, 2.0),
    # every sequence dense at the same length: equal segments of N tiles
    ("all_dense_equal", C0.scaled(batch=5, seq_len=700), [700] * 5, 30, 0.5),
    # equal segments of one block each (fewer tiles than a CTA's minimum)
    ("equal_one_block", C3.scaled(batch=9, seq_len=640, layers=1), [640] * 9, 1, 2.0),
], ids=lambda v: v if isinstance(v, str) else "")
def test_decode_split_of_equal_segments(K, name, w, lens, k, gamma):
    x = to_dev(generate_layer(w, 0, seq_lens=lens), "cuda:0")
    dec, *_ = _run(K, w, x, k, gamma=gamma)
    for b, T in enumerate(lens):
        if T == 0:
            assert int(dec.n_sel[b]) == 0
            assert torch.all(dec.out[b] == 0) and torch.all(torch.isneginf(dec.lse[b]))
        else:
            check_sequence(dec, x, b, T, w.block_size, k, dec.scale, gamma=gamma)
    if name == "all_dense_equal":
        assert bool(dec.dense_flag.all())


def test_bad_block_table_is_latched_not_fatal(K):
    w = C0.scaled(batch=2, seq_len=320)
    x = to_dev(generate_layer(w, 0), "cuda:0")
    x["block_table"][1, 3] = 10 ** 6
    dec = _decoder(w, x)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS
    assert K.kvsel_get_error() == 0   # read-and-clear


def test_oversized_k_is_clamped_and_latched(K):
    w = C0.scaled(batch=1, seq_len=320)
    x = to_dev(generate_layer(w, 0), "cuda:0")
    dec = _decoder(w, x, k_max=8)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.fill_(12)
    dec.select(x["q"], summ, x["seq_lens"])
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS
    assert int(dec.n_sel[0]) == 8


# ---------------------------------------------------------- full sizes ---

def _full_layer(K, w, k, layer=0, sample=None, gamma=2.0):
    x = generate_layer(w, layer, device="cuda:0", perm=True)
    dec, summ, _, scores = _run(K, w, x, k, gamma=gamma)
    verdicts = []
    bs = range(w.batch) if sample is None else sample
    for b in bs:
        v, emax, emean = check_sequence(dec, x, b, w.seq_len, w.block_size, k, dec.scale,
                                        scores_gpu=scores, summaries_gpu=summ, gamma=gamma)
        verdicts.append(v)
    return dec, x, verdicts


def test_c0_full(K):
    _full_layer(K, C0, 16)


@pytest.mark.parametrize("keep", C1.keep)
def test_c1_opt67b_needles_selected(K, keep):
    k = C1.k_for(keep)
    dec, x, v = _full_layer(K, C1, k, layer=0)
    for b in range(C1.batch):
        sel = set(dec.sel_idx[b, : int(dec.n_sel[b])].cpu().tolist())
        assert set(C1.needles) <= sel


def test_c2_minicpm_gqa16(K):
    _full_layer(K, C2, C2.k_for(C2.keep[0]))


def test_c3_qwen3_4b_batch16(K):
    _full_layer(K, C3, C3.k_for(C3.keep[0]))


def test_c4_offload_tier_fetch_then_decode(K):
    """Full C4 shape at the 5 % Minimum Keep Floor: K/V in pinned host memory,
    summaries on the GPU, the selected spans fetched over the host link,
    attention over the staging buffer; every sequence against the oracle
    (selection under the tie rule, no sequence dense at this keep ratio, and
    attention). The dense fallback of the host tier is checked by
    test_offload_staged_dense_fallback_mixed."""
    w = C4
    k = w.k_for(w.keep_floor)
    x = generate_layer(w, 0, device="cuda:0", perm=False)
    N = w.n_blocks
    page = tuple(x["kv_pages"].shape[1:])
    host = torch.empty((w.batch, N) + page, dtype=torch.bfloat16, pin_memory=True)
    host_tier_layout(x["kv_pages"], x["block_table"], N, out=host)
    dec = _decoder(w, x, k_max=N)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    del x["kv_pages"]
    torch.cuda.empty_cache()
    dec.k_per_seq.fill_(k)
    dec.select(x["q"], summ, x["seq_lens"], gamma=w.gamma)
    slots = k
    staging = torch.empty((w.batch, slots) + page, dtype=torch.bfloat16, device="cuda:0")
    from query_aware_sparse_block_gb300 import kvsel as KK
    kv = KK.kv_host(host, N, staging, slots)
    dec.attend(x["q"], kv, x["seq_lens"])
    torch.cuda.synchronize()
    for b in range(w.batch):
        qb = bits(x["q"][b])
        kb = bits(natural_blocks(host[b, :, :, 0]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
        vb = bits(natural_blocks(host[b, :, :, 1]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
        sb, _, _ = o.block_summaries(kb, w.seq_len, w.block_size)
        sc = o.block_scores(qb, sb)
        gsel = dec.sel_idx[b, : int(dec.n_sel[b])].cpu().numpy()
        selection_verdict(sc, k, gsel)
        assert not bool(dec.dense_flag[b])
        ref, _ = o.attend(qb, kb, vb, o.tokens_of_blocks(gsel, w.seq_len, w.block_size), dec.scale)
        emax, emean = attn_errors(dec.out[b].cpu().numpy(), ref)
        assert emax <= 1e-2 and emean <= 1e-3, (b, emax, emean)
    # staging slot o holds the page of the o-th selected block
    b = 7
    gsel = dec.sel_idx[b, : int(dec.n_sel[b])].cpu()
    assert torch.equal(staging[b, :5].cpu(), host[b, gsel[:5].long()])


def test_offload_staged_dense_fallback_mixed(K):
    """The host tier through KVSEL_KV_HOST (the selected spans, or every block
    of a dense sequence, gathered into staging, then attended) with the gamma
    rule deciding per sequence ("SparPR KV cache recovery on a consumer GPU",
    paragraph "On-demand local recomputation with cost-aware fallback": once
    the sparse path is no longer clearly cheaper, recover everything). The
    copy/recompute model gives r = 1 for the C4 shape with GB300-class link and
    compute rates, so k = N and every sequence of C4 is dense; here the same
    shape at a reduced batch and length mixes k = N with keep ratios above and
    below gamma = 0.8, over ragged lengths. Dense sequences must equal full
    attention, the others attention over their selection."""
    w = C4
    r = K.kvsel_budget(w.block_size, w.n_kvheads, w.head_dim, 2, w.hidden, w.n_blocks, 211e9, 1.7376e15,
                       keep_floor=w.keep_floor, gamma=w.gamma)
    assert r.r == 1.0 and r.k == w.n_blocks and r.dense == 1
    ws = w.scaled(batch=6, seq_len=8192)
    lens = [8192, 8192, 5000, 8192, 64, 7000]
    ks = [128, 13, 79, 90, 1, 100]               # N = 128, 128, 79, 128, 1, 110
    dense_want = [True, False, True, False, True, True]
    x = generate_layer(ws, 0, device="cuda:0", perm=True, seq_lens=lens)
    N = x["max_blocks"]
    page = tuple(x["kv_pages"].shape[1:])
    host = torch.empty((ws.batch, N) + page, dtype=torch.bfloat16, pin_memory=True)
    host_tier_layout(x["kv_pages"], x["block_table"], N, out=host)
    dec = _decoder(ws, x, k_max=N)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.copy_(torch.tensor(ks, dtype=torch.int32))
    dec.select(x["q"], summ, x["seq_lens"], gamma=ws.gamma)
    staging = torch.empty((ws.batch, N) + page, dtype=torch.bfloat16, device="cuda:0")
    staging.fill_(float("nan"))                  # every attended slot must be written by the fetch
    from query_aware_sparse_block_gb300 import kvsel as KK
    dec.attend(x["q"], KK.kv_host(host, N, staging, N), x["seq_lens"])
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == 0
    assert [bool(v) for v in dec.dense_flag.cpu()] == dense_want
    for b in range(ws.batch):
        check_sequence(dec, x, b, lens[b], ws.block_size, ks[b], dec.scale, gamma=ws.gamma)
    # a dense sequence's staging holds all its blocks in order
    assert torch.equal(staging[2, :79].cpu(), host[2, :79])
