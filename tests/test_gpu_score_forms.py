"""The two forms of the score + Top-k call give the same results bit for bit.

kvsel_score_topk (and its append / window variants) runs either as one launch
of thread-block clusters (one cluster per sequence; the leader CTA ranks the
keys its peers wrote into its shared memory) or as a score grid followed by a
Top-k grid. Both compute every block score with the same fp32 operations in
the same order ("SparPR KV cache recovery on a consumer GPU", paragraph
"Query-Aware key-block selection": score = sum over heads of query . block
summary; Top-k with ties to the lower index; spans and the gamma rule of
paragraph "On-demand local recomputation with cost-aware fallback"). Here both
forms run on the same inputs and every output is compared bit for bit: the
fp32 scores, the selection, the spans, the counts and the dense flags, and
with a folded append also the pages, summaries and fp64 accumulators it
writes. The cluster form is checked against the oracle by the parity tests,
which take it by default.

The shapes cover every per-lane vector count of the scoring kernels (1, 2, 4,
16 vectors of 8 channels per lane), 8 and 16 lanes per block as well as 32,
ragged and empty sequences, a partial last block, windows, a folded append,
clustered and tied scores, and a batch of 64 sequences of 2048 blocks.
"""
from __future__ import annotations

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
    yield kvsel
    kvsel.kvsel_set_score_path(kvsel.KVSEL_SCORE_PATH_AUTO)


def _decoder(batch, Hq, Hkv, d, B, max_blocks, k_max):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    return SparseDecoder(batch, Hq, Hkv, d, B, max_blocks, k_max=k_max, device="cuda:0")


def _outputs(dec, scores, N):
    n = dec.n_sel.cpu().numpy()
    ns = dec.n_spans.cpu().numpy()
    out = dict(n_sel=n.copy(), n_spans=ns.copy(), dense=dec.dense_flag.cpu().numpy().copy())
    out["sel"] = [dec.sel_idx[b, : n[b]].cpu().numpy().copy() for b in range(len(n))]
    out["st"] = [dec.span_start[b, : ns[b]].cpu().numpy().copy() for b in range(len(ns))]
    out["ln"] = [dec.span_len[b, : ns[b]].cpu().numpy().copy() for b in range(len(ns))]
    if scores is not None:
        s = scores.cpu()
        out["scores"] = [s[b, : N[b]].view(torch.int32).numpy().copy() for b in range(len(N))]
    return out


def _assert_same(x, y):
    assert x.keys() == y.keys()
    for k in x:
        if isinstance(x[k], list):
            assert len(x[k]) == len(y[k])
            for i, (u, v) in enumerate(zip(x[k], y[k])):
                assert np.array_equal(u, v), f"{k} differs in sequence {i}"
        else:
            assert np.array_equal(x[k], y[k]), f"{k} differs"


def _both_forms(K, dec, run, N, with_scores=True, with_append=False):
    """run(scores) enqueues the call; returns the two forms' outputs."""
    form, ctas = K.kvsel_score_path_for(dec.p, with_append)
    assert form == K.KVSEL_SCORE_PATH_CLUSTER and ctas >= 1, "the cluster form does not take this shape"
    res = []
    for path in (K.KVSEL_SCORE_PATH_TWO_GRID, K.KVSEL_SCORE_PATH_CLUSTER):
        K.kvsel_set_score_path(path)
        for t in (dec.sel_idx, dec.span_start, dec.span_len):
            t.fill_(-7)
        dec.n_sel.fill_(-1)
        dec.n_spans.fill_(-1)
        dec.dense_flag.fill_(9)
        scores = None
        if with_scores:
            scores = torch.full((dec.p.batch, dec.p.max_blocks), float("nan"), device="cuda:0")
        run(scores)
        torch.cuda.synchronize()
        assert K.kvsel_get_error() == 0
        res.append(_outputs(dec, scores, N))
    K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_AUTO)
    return res


def _random_inputs(batch, Hq, Hkv, d, max_blocks, seed, scale=1.0):
    g = torch.Generator(device="cuda:0")
    g.manual_seed(seed)
    q = torch.randn((batch, Hq, d), generator=g, device="cuda:0").to(torch.bfloat16)
    summ = (torch.randn((batch, max_blocks, Hkv, d), generator=g, device="cuda:0") * scale).to(torch.bfloat16)
    return q, summ


CASES = [
    # name, batch, Hq, Hkv, d, B, max_blocks, lens (tokens), ks
    ("c0_mha_d64", 1, 8, 8, 64, 16, 64, [1024], [16]),
    ("c1_mha_d128_keep50", 4, 32, 32, 128, 16, 256, [4096] * 4, [128] * 4),
    ("c1_mha_d128_keep10_ragged", 4, 32, 32, 128, 16, 256, [4096, 17, 0, 4000], [26, 26, 5, 26]),
    ("c2_gqa_kv2", 1, 32, 2, 128, 64, 2048, [131072], [64]),
    ("c3_gqa_kv8", 16, 32, 8, 128, 32, 1024, [32768 - 7] * 16, [128] * 16),
    ("c3_ragged", 5, 32, 8, 128, 32, 1024, [32768, 1, 2047, 0, 20000], [128, 1, 40, 7, 128]),
    ("c4_batch64", 64, 32, 2, 128, 64, 2048, [131072] * 64, [102] * 64),
    ("kv1_d64_lanes8", 3, 4, 1, 64, 16, 313, [5000, 4999, 16], [40, 313, 1]),
    ("kv1_d128_lanes16", 3, 16, 1, 128, 16, 700, [11200, 333, 11199], [70, 20, 700]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_forms_agree_bit_for_bit(K, case):
    name, batch, Hq, Hkv, d, B, mb, lens, ks = case
    dec = _decoder(batch, Hq, Hkv, d, B, mb, k_max=max(ks))
    q, summ = _random_inputs(batch, Hq, Hkv, d, mb, seed=len(name) * 7919 + batch)
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda:0")
    dec.k_per_seq.copy_(torch.tensor(ks, dtype=torch.int32))
    N = [(t + B - 1) // B for t in lens]
    for gamma, tau in ((2.0, 0.0), (0.5, 0.25)):
        a, c = _both_forms(K, dec, lambda sc: dec.select(q, summ, seq_lens, gamma=gamma, tau_rel=tau,
                                                         scores_out=sc), N)
        _assert_same(a, c)
        for b in range(batch):
            assert a["n_sel"][b] == min(ks[b], N[b])
    # without a score output
    a, c = _both_forms(K, dec, lambda sc: dec.select(q, summ, seq_lens, gamma=0.9), N, with_scores=False)
    _assert_same(a, c)


def test_forms_agree_on_tied_and_clustered_scores(K):
    """Summaries with one non-zero channel and a one-hot query make every
    score a chosen bf16 value: few distinct values, all equal, adjacent
    floating-point values, NaN and infinities."""
    batch, mb = 6, 2000
    dec = _decoder(batch, 1, 1, 64, 16, mb, k_max=mb)
    rng = np.random.default_rng(5)
    rows = [rng.integers(-3, 4, mb).astype(np.float32),
            np.full(mb, 0.75, np.float32),
            (1.0 + rng.integers(0, 128, mb) / 128.0).astype(np.float32),
            rng.standard_normal(mb).astype(np.float32),
            np.concatenate([[np.nan, 1.0, -np.inf, 2.0, np.inf], rng.standard_normal(mb - 5)]).astype(np.float32),
            (rng.standard_normal(mb) * 1e-4).astype(np.float32)]
    summ = torch.zeros((batch, mb, 1, 64), dtype=torch.bfloat16)
    for b, r in enumerate(rows):
        summ[b, :, 0, 0] = torch.from_numpy(r).to(torch.bfloat16)
    summ = summ.to("cuda:0")
    q = torch.zeros((batch, 1, 64), dtype=torch.bfloat16, device="cuda:0")
    q[:, 0, 0] = 1.0
    lens = [mb * 16, mb * 16 - 5, 16 * 1500, mb * 16, mb * 16, 16 * 999 + 1]
    ks = [mb // 8, 100, 1500 - 1, 1, mb - 3, 500]
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda:0")
    dec.k_per_seq.copy_(torch.tensor(ks, dtype=torch.int32))
    N = [(t + 15) // 16 for t in lens]
    a, c = _both_forms(K, dec, lambda sc: dec.select(q, summ, seq_lens, gamma=0.7, scores_out=sc), N)
    _assert_same(a, c)


@pytest.mark.parametrize("window", [(0, 0), (1, 4), (3, 0), (0, 9)])
def test_forms_agree_with_windows(K, window):
    batch, mb = 5, 1024
    dec = _decoder(batch, 32, 8, 128, 32, mb, k_max=140)
    q, summ = _random_inputs(batch, 32, 8, 128, mb, seed=11 + sum(window))
    lens = [32768, 100, 2047, 0, 320]
    ks = [128, 3, 40, 7, 131]
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda:0")
    dec.k_per_seq.copy_(torch.tensor(ks, dtype=torch.int32))
    N = [(t + 31) // 32 for t in lens]
    a, c = _both_forms(K, dec, lambda sc: dec.select_window(q, summ, seq_lens, *window, gamma=0.6,
                                                            scores_out=sc), N)
    _assert_same(a, c)


def test_forms_agree_with_folded_append(K):
    """kvsel_append_score_topk through both forms from the same state: every
    output, and the pages, summaries and accumulators the append writes."""
    from query_aware_sparse_block_gb300 import kvsel as KV
    w = C3.scaled(batch=6, seq_len=4096, layers=1)
    lens0 = [4096 - 1, 31, 32, 0, 4000, 1]         # tokens before the append
    x = {k: (v.to("cuda:0") if torch.is_tensor(v) else v)
         for k, v in generate_layer(w, 0, seq_lens=lens0).items()}
    mb = x["max_blocks"]
    dec = _decoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, mb, k_max=64)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    g = torch.Generator(device="cuda:0")
    g.manual_seed(77)
    shape = (w.batch, w.n_kvheads, w.head_dim)
    new_k = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
    new_v = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
    pos = torch.tensor([t if b != 3 else -1 for b, t in enumerate(lens0)], dtype=torch.int32, device="cuda:0")
    lens1 = [t + 1 if b != 3 else t for b, t in enumerate(lens0)]
    seq_lens = torch.tensor(lens1, dtype=torch.int32, device="cuda:0")
    dec.k_per_seq.copy_(torch.tensor([64, 1, 2, 5, 60, 1], dtype=torch.int32))
    N = [(t + w.block_size - 1) // w.block_size for t in lens1]
    state0 = (x["kv_pages"].clone(), summ.clone(), acc.clone())
    states = []

    def run(sc):
        x["kv_pages"].copy_(state0[0])
        summ.copy_(state0[1])
        acc.copy_(state0[2])
        dec.append_select(x["kv_pages"], x["block_table"], pos, x["q"], summ, acc, seq_lens,
                          new_k=new_k, new_v=new_v, gamma=0.8, scores_out=sc)
        torch.cuda.synchronize()
        states.append((x["kv_pages"].view(torch.int16).clone(), summ.view(torch.int16).clone(),
                       acc.view(torch.int64).clone()))

    a, c = _both_forms(KV, dec, run, N, with_append=True)
    _assert_same(a, c)
    for u, v in zip(states[0], states[1]):
        assert torch.equal(u, v)


def test_cluster_form_rejects_what_it_cannot_take(K):
    """A key row longer than the leader's shared memory holds goes through the
    two-grid form under AUTO and fails with UNSUPPORTED when the cluster form
    is forced."""
    p = K.problem(2, 8, 8, 64, 16, 16384, 64)
    assert K.kvsel_score_path_for(p)[0] == K.KVSEL_SCORE_PATH_TWO_GRID
    dec = _decoder(2, 8, 8, 64, 16, 16384, k_max=64)
    q, summ = _random_inputs(2, 8, 8, 64, 16384, seed=3)
    seq_lens = torch.tensor([16384 * 16, 5], dtype=torch.int32, device="cuda:0")
    dec.k_per_seq.fill_(64)
    K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_CLUSTER)
    try:
        with pytest.raises(K.KvselError) as ei:
            dec.select(q, summ, seq_lens)
        assert ei.value.code == K.KVSEL_ERR_UNSUPPORTED
    finally:
        K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_AUTO)
    dec.select(q, summ, seq_lens)
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == 0
    assert int(dec.n_sel[0]) == 64 and int(dec.n_sel[1]) == 1
