"""GPU: prefetch into the block cache of the host tier (kvsel_cache_prefetch)
and the Top-k on given score rows that predicts what to prefetch
(kvsel_select_scores).

  * The cache state and the copied pages after every prefetch and every step
    equal the oracle's BlockCache bit for bit, on random predictions that
    keep, drop and add blocks and sometimes name the block holding the last
    token.
  * kvsel_select_scores equals the oracle's Top-k, span merge and dense rule
    on score rows built to have exact ties, infinities, NaN and ragged
    lengths, and equals the selection of kvsel_score_topk on that call's own
    score rows.
  * Layer-ahead prefetch on a second stream ("KV cache offloading": the
    Hugging Face Transformers paragraph and section "SparDA"): while layer l
    selects, fetches and attends on the compute stream, the next layer's
    cache is loaded on a copy stream with that layer's Top-(k+m) of its
    previous step. On a MiniCPM-shaped host tier with drifting queries the
    attention equals the path without prefetch bit for bit and the oracle,
    every cache state equals the oracle's BlockCache, and the compute
    stream's fetches copy fewer blocks.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as o
from tests._parity import attn_errors
from workloads import C0, C4
from workloads.generate import bits, generate_layer, host_tier_layout, natural_blocks

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


def _check_state(cache, ref, b, N, slots, tag):
    assert cache.block_in[b].cpu().tolist() == ref.block_in, tag
    assert cache.last_use[b].cpu().tolist() == ref.last_use, tag
    want = torch.full((N,), -1, dtype=torch.int32)
    for blk, s in ref.slot_of.items():
        want[blk] = b * slots + s
    assert torch.equal(cache.page_of[b].cpu(), want), tag


def _as_rows(lists, width):
    t = torch.zeros((len(lists), width), dtype=torch.int32)
    for b, l in enumerate(lists):
        t[b, : len(l)] = torch.from_numpy(np.asarray(l, dtype=np.int32))
    n = torch.tensor([len(l) for l in lists], dtype=torch.int32)
    return t.to("cuda:0"), n.to("cuda:0")


@pytest.mark.parametrize("slots,locality", [(12, 0.7), (16, 0.4)])
def test_prefetch_state_and_pages_match_the_oracle(K, slots, locality):
    from query_aware_sparse_block_gb300.runtime import HostBlockCache, SparseDecoder
    w = C0.scaled(batch=3, seq_len=64 * 16)
    N, k, k_max = 64, 6, 12
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, N, k_max=k_max,
                        device="cuda:0")
    page = (w.n_kvheads, 2, w.head_dim // 64, w.block_size, 64)
    g = torch.Generator().manual_seed(slots)
    host = torch.randn((w.batch, N) + page, generator=g).to(torch.bfloat16).pin_memory()
    cache = HostBlockCache(dec, slots, page)
    seq_lens = torch.full((w.batch,), N * w.block_size, dtype=torch.int32, device="cuda:0")
    ref = [o.BlockCache(slots) for _ in range(w.batch)]
    rng = np.random.default_rng(slots)
    prev = [np.array([], dtype=np.int64)] * w.batch
    prefetched = 0
    for step in range(30):
        # a prediction per sequence: most of the last selection, other blocks,
        # sometimes the block holding the last token
        preds = []
        for b in range(w.batch):
            extra = rng.choice(N, size=int(rng.integers(0, k_max - k + 1)), replace=False)
            pred = np.union1d(prev[b][rng.random(len(prev[b])) < 0.8], extra)
            if step % 4 == 1:
                pred = np.union1d(pred, [N - 1])
            preds.append(pred[:k_max])
        pi, pn = _as_rows(preds, k_max)
        cache.prefetch(host, N, seq_lens, pi, pn)
        torch.cuda.synchronize()
        npf = cache.n_prefetched.cpu().tolist()
        for b in range(w.batch):
            jobs = ref[b].prefetch(preds[b], N - 1)
            assert npf[b] == len(jobs), (step, b)
            prefetched += len(jobs)
            _check_state(cache, ref[b], b, N, slots, ("prefetch", step, b))
        # the step: a selection drawn around the prediction
        sels = []
        for b in range(w.batch):
            keep = preds[b][rng.random(len(preds[b])) < locality]
            rest = np.setdiff1d(np.arange(N), keep)
            kk = int(rng.integers(1, k + 1))
            sel = np.sort(np.concatenate([keep[:kk], rng.choice(rest, size=kk - min(kk, len(keep)),
                                                                 replace=False)]))
            sels.append(sel)
        si, sn = _as_rows(sels, k_max)
        cache.fetch(host, N, seq_lens, si, sn)
        torch.cuda.synchronize()
        nf = cache.n_fetched.cpu().tolist()
        for b in range(w.batch):
            jobs, _ = ref[b].step(sels[b], step, N - 1)
            assert nf[b] == len(jobs), (step, b)
            _check_state(cache, ref[b], b, N, slots, ("step", step, b))
            for blk, s in ref[b].slot_of.items():
                assert torch.equal(cache.pool[b * slots + s].cpu().view(torch.int16),
                                   host[b, blk].view(torch.int16)), (step, b, blk)
        prev = sels
    assert prefetched > 0


def test_prefetch_rejects_a_prediction_that_is_not_ascending(K):
    from query_aware_sparse_block_gb300.runtime import HostBlockCache, SparseDecoder
    w = C0.scaled(batch=1, seq_len=320)
    dec = SparseDecoder(1, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, 20, k_max=4,
                        device="cuda:0")
    page = (w.n_kvheads, 2, w.head_dim // 64, w.block_size, 64)
    host = torch.zeros((1, 20) + page, dtype=torch.bfloat16).pin_memory()
    cache = HostBlockCache(dec, 4, page)
    pred = torch.tensor([[5, 2, 8, 11]], dtype=torch.int32, device="cuda:0")
    cache.prefetch(host, 20, torch.tensor([320], dtype=torch.int32, device="cuda:0"), pred,
                   torch.tensor([4], dtype=torch.int32, device="cuda:0"))
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS
    # the entries that break the order are not served; 19 is the last block
    assert sorted(b for b in cache.block_in[0].cpu().tolist() if b >= 0) == [5, 8, 11]
    assert sorted(cache.last_use[0].cpu().tolist()) == [-1] * 4


def _score_rows(rng, batch, max_blocks):
    """Rows with exact ties (small integers), infinities and NaN."""
    rows = rng.integers(-6, 7, size=(batch, max_blocks)).astype(np.float32)
    rows[0, ::7] = np.inf
    rows[0, 3::11] = -np.inf
    rows[1, 5::9] = np.nan
    rows[2] = 0.0                                    # every score tied
    rows[3] = rng.standard_normal(max_blocks).astype(np.float32)
    return rows


@pytest.mark.parametrize("max_blocks", [64, 1000, 4096])
def test_select_scores_equals_the_oracle(K, max_blocks):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    rng = np.random.default_rng(max_blocks)
    batch, B = 6, 16
    k_max = min(max_blocks, 300)
    dec = SparseDecoder(batch, 8, 8, 64, B, max_blocks, k_max=k_max, device="cuda:0")
    rows = _score_rows(rng, batch, max_blocks)
    # ragged lengths: full, partial last block, one token, nothing
    T = [max_blocks * B, max_blocks * B - 5, (max_blocks // 3) * B + 1, max_blocks * B, 1, 0]
    ks = [k_max, 17, max_blocks, 1, 3, 5]             # k above N and above k_max included
    seq_lens = torch.tensor(T, dtype=torch.int32, device="cuda:0")
    k_per_seq = torch.tensor([min(k, k_max) for k in ks], dtype=torch.int32, device="cuda:0")
    scores = torch.from_numpy(rows).to("cuda:0")
    gamma, tau_rel = 0.625, 1.5                      # exact in fp32 and fp64
    K.kvsel_select_scores(dec.p, scores, seq_lens, k_per_seq, dec.sel_idx, dec.n_sel, dec.span_start,
                          dec.span_len, dec.n_spans, gamma=gamma, tau_rel=tau_rel,
                          dense_flag=dec.dense_flag)
    torch.cuda.synchronize()
    for b in range(batch):
        N = (T[b] + B - 1) // B
        k = min(ks[b], k_max)
        sel = o.topk_blocks(rows[b, :N].astype(np.float64), k) if N else np.array([], dtype=np.int64)
        starts, lens = o.merge_spans(sel)
        n = int(dec.n_sel[b])
        assert dec.sel_idx[b, :n].cpu().tolist() == [int(v) for v in sel], b
        ns = int(dec.n_spans[b])
        assert dec.span_start[b, :ns].cpu().tolist() == [int(v) for v in starts], b
        assert dec.span_len[b, :ns].cpu().tolist() == [int(v) for v in lens], b
        want_dense = bool(N) and o.dense_fallback(len(starts), len(sel), N, gamma, tau_rel)
        assert bool(dec.dense_flag[b]) == want_dense, b


def test_select_scores_reproduces_the_score_call_selection(K):
    """kvsel_select_scores on the rows a kvsel_score_topk call wrote gives
    that call's selection, spans and flag bit for bit, under both forms."""
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    w = C0.scaled(batch=5, seq_len=2048)
    x = generate_layer(w, 0, device="cuda:0")
    mb = w.n_blocks
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, mb, k_max=40,
                        device="cuda:0")
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    seq_lens = torch.tensor([2048, 2000, 17, 1, 1500], dtype=torch.int32, device="cuda:0")
    k_per_seq = torch.tensor([40, 13, 2, 1, 29], dtype=torch.int32, device="cuda:0")
    scores = torch.empty((w.batch, mb), dtype=torch.float32, device="cuda:0")
    two = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, mb, k_max=40,
                        device="cuda:0")
    for path in (K.KVSEL_SCORE_PATH_TWO_GRID, K.KVSEL_SCORE_PATH_CLUSTER):
        prev = K.kvsel_set_score_path(path)
        try:
            dec.select(x["q"], summ, seq_lens, k_per_seq=k_per_seq, gamma=0.5, scores_out=scores)
        finally:
            K.kvsel_set_score_path(prev)
        K.kvsel_select_scores(two.p, scores, seq_lens, k_per_seq, two.sel_idx, two.n_sel,
                              two.span_start, two.span_len, two.n_spans, gamma=0.5,
                              dense_flag=two.dense_flag)
        torch.cuda.synchronize()
        for name in ("n_sel", "n_spans", "dense_flag"):
            assert torch.equal(getattr(dec, name), getattr(two, name)), (path, name)
        for b in range(w.batch):
            n, ns = int(dec.n_sel[b]), int(dec.n_spans[b])
            assert torch.equal(dec.sel_idx[b, :n], two.sel_idx[b, :n]), (path, b)
            assert torch.equal(dec.span_start[b, :ns], two.span_start[b, :ns]), (path, b)
            assert torch.equal(dec.span_len[b, :ns], two.span_len[b, :ns]), (path, b)


def test_layer_ahead_prefetch_on_a_second_stream(K):
    """Two MiniCPM4.1-8B-shaped layers (32 q / 2 KV heads, d 128, 131072
    tokens in blocks of 64) for 4 sequences, each with its own host tier and
    drifting queries (q_s = 0.95 q_(s-1) + 0.31 e_s). Per step and layer on
    the compute stream: select (scores kept), fetch, attend. On the copy
    stream, once layer l's fetch is done: the Top-(k + m) of layer l+1's
    previous scores is prefetched into layer l+1's cache (layer 0 of the
    next step after the last layer)."""
    from query_aware_sparse_block_gb300.runtime import BlockPredictor, HostBlockCache, SparseDecoder
    w = C4.scaled(batch=4)
    N = w.n_blocks
    k = w.k_for(w.keep_floor)
    m = k // 2
    L = 2
    dev = "cuda:0"
    layers = []
    for l in range(L):
        x = generate_layer(w, l, device=dev, perm=False)
        page = tuple(x["kv_pages"].shape[1:])
        host = torch.empty((w.batch, N) + page, dtype=torch.bfloat16, pin_memory=True)
        host_tier_layout(x["kv_pages"], x["block_table"], N, out=host)
        dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, N, k_max=k + m,
                            device=dev)
        summ, acc = dec.new_summaries()
        dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
        dec.k_per_seq.fill_(k)
        plain = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, N, k_max=k + m,
                              device=dev)
        layers.append(dict(
            x=dict(q=x["q"], seq_lens=x["seq_lens"]), host=host, dec=dec, summ=summ, plain=plain,
            cache=HostBlockCache(dec, 2 * (k + m), page), ref_cache=HostBlockCache(plain, 2 * (k + m), page),
            pred=BlockPredictor(dec, k + m), scores=torch.empty((w.batch, N), dtype=torch.float32, device=dev),
            oref=[o.BlockCache(2 * (k + m)) for _ in range(w.batch)],
            oplain=[o.BlockCache(2 * (k + m)) for _ in range(w.batch)], q=x["q"].float(),
            g=torch.Generator(device=dev).manual_seed(500 + l), have_scores=False))
        del x
        torch.cuda.empty_cache()
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    crit = {"with": 0, "without": 0}
    for step in range(5):
        for l in range(L):
            Ly = layers[l]
            if step:
                Ly["q"] = 0.95 * Ly["q"] + math.sqrt(1 - 0.95 ** 2) * torch.randn(
                    Ly["q"].shape, generator=Ly["g"], device=dev)
            qb = Ly["q"].to(torch.bfloat16)
            dec, cache = Ly["dec"], Ly["cache"]
            dec.select(qb, Ly["summ"], Ly["x"]["seq_lens"], scores_out=Ly["scores"])
            if "prefetched" in Ly:
                compute.wait_event(Ly.pop("prefetched"))
            cache.fetch(Ly["host"], N, Ly["x"]["seq_lens"], dec.sel_idx, dec.n_sel)
            fetched = torch.cuda.Event()
            fetched.record(compute)
            dec.attend(qb, cache.kv, Ly["x"]["seq_lens"], use_dense_flag=False)
            # the same selection without prefetch
            plain = Ly["plain"]
            for name in ("sel_idx", "n_sel", "span_start", "span_len", "n_spans"):
                getattr(plain, name).copy_(getattr(dec, name))
            Ly["ref_cache"].fetch(Ly["host"], N, Ly["x"]["seq_lens"], plain.sel_idx, plain.n_sel)
            plain.attend(qb, Ly["ref_cache"].kv, Ly["x"]["seq_lens"], use_dense_flag=False)
            # the next layer's prefetch on the copy stream, from its previous scores
            nl = (l + 1) % L
            Nx = layers[nl]
            if Nx["have_scores"]:
                copy.wait_event(fetched)
                with torch.cuda.stream(copy):
                    Nx["pred"].from_scores(Nx["scores"], Nx["x"]["seq_lens"], stream=copy)
                    Nx["cache"].prefetch(Nx["host"], N, Nx["x"]["seq_lens"], Nx["pred"].pred_idx,
                                         Nx["pred"].n_pred, stream=copy)
                ev = torch.cuda.Event()
                ev.record(copy)
                Nx["prefetched"] = ev
            torch.cuda.synchronize()
            Ly["have_scores"] = True
            assert torch.equal(dec.out, plain.out) and torch.equal(dec.lse, plain.lse), (step, l)
            nf = cache.n_fetched.cpu().tolist()
            crit["with"] += sum(nf)
            crit["without"] += sum(Ly["ref_cache"].n_fetched.cpu().tolist())
            for b in range(w.batch):
                gsel = dec.sel_idx[b, : int(dec.n_sel[b])].cpu().numpy()
                jobs, _ = Ly["oref"][b].step(gsel, step, N - 1)
                assert nf[b] == len(jobs), (step, l, b)
                _check_state(cache, Ly["oref"][b], b, N, 2 * (k + m), ("step", step, l, b))
                Ly["oplain"][b].step(gsel, step, N - 1)
            if Nx["have_scores"] and "prefetched" in Nx:
                # the prediction and the prefetched state against the oracle
                sc = Nx["scores"].cpu().numpy().astype(np.float64)
                npf = Nx["cache"].n_prefetched.cpu().tolist()
                for b in range(w.batch):
                    want = o.topk_blocks(sc[b], k + m)
                    got = Nx["pred"].pred_idx[b, : int(Nx["pred"].n_pred[b])].cpu().numpy()
                    assert got.tolist() == want.tolist(), (step, l, b)
                    jobs = Nx["oref"][b].prefetch(want, N - 1)
                    assert npf[b] == len(jobs), (step, l, b)
                    _check_state(Nx["cache"], Nx["oref"][b], b, N, 2 * (k + m), ("prefetch", step, nl, b))
            if step == 4 and l == 1:
                b = 2
                host = Ly["host"]
                qbits = bits(qb[b])
                kb = bits(natural_blocks(host[b, :, :, 0]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
                vb = bits(natural_blocks(host[b, :, :, 1]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
                gsel = dec.sel_idx[b, : int(dec.n_sel[b])].cpu().numpy()
                ref, _ = o.attend(qbits, kb, vb, o.tokens_of_blocks(gsel, w.seq_len, w.block_size), dec.scale)
                emax, emean = attn_errors(dec.out[b].cpu().numpy(), ref)
                assert emax <= 1e-2 and emean <= 1e-3, (emax, emean)
    # the compute stream's fetches carried fewer blocks with the prefetch
    assert crit["with"] < crit["without"], crit
