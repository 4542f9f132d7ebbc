"""Top-k threshold search on scores chosen exactly.

The summaries carry one non-zero channel (KV head 0, channel 0) and the query
is the unit vector on that channel, so every block score equals a bf16 value
picked here: heavy ties, all-equal rows, runs of adjacent floating-point
values (the search must narrow down to a single key value), ties that
straddle the k-th score, rows short enough to be ranked directly, and rows of
16384 blocks. Selection, spans and the dense flag must equal the oracle's
Top-k (ties to the lower index, "SparPR KV cache recovery on a consumer GPU",
paragraph "Query-Aware key-block selection") bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as o

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


def _rows(rng, nmax):
    """Rows of at most nmax blocks; (scores, k) pairs."""
    n = lambda x: min(x, nmax)
    adj = (1.0 + rng.integers(0, 128, n(5000)) / 128.0).astype(np.float32)       # adjacent bf16 values
    h = n(3000) // 2
    mixed = np.concatenate([rng.standard_normal(h) * 1e-4, rng.standard_normal(h) * 1e3])
    m = n(3000)
    straddle = np.full(m, -1.0); straddle[: m // 15] = 5.0
    straddle[rng.choice(m, m // 7, replace=False)] = 2.0
    return [
        (rng.integers(-3, 4, nmax).astype(np.float64), nmax // 8),  # 7 distinct values
        (np.full(nmax, 0.75), 100),                                 # all equal
        (adj.astype(np.float64), n(5000) // 6),
        (rng.standard_normal(n(3000)), n(3000) // 8),
        (mixed, len(mixed) // 10),
        (straddle, int((straddle > 2).sum()) + m // 20),            # ties at the k-th value straddle it
        (rng.integers(0, 3, 100).astype(np.float64), 37),           # short row: direct ranking
        (np.array([1.5]), 1),
        (rng.standard_normal(7), 0),
        (rng.standard_normal(129), 128),
        (rng.standard_normal(nmax), nmax - 1),
        (rng.standard_normal(nmax - 37), 1),
        # non-finite scores: NaN of either sign ranks below -inf, ties by index
        (np.concatenate([[np.nan, 1.0, -np.inf, -np.nan, 2.0, np.inf, np.nan],
                         rng.standard_normal(n(200) - 7)]), n(200) - 3),
    ]


@pytest.mark.parametrize("max_blocks", [1000, 2048, 4096, 4097, 16384])
def test_threshold_search_paths_match_oracle(K, max_blocks):
    """Rows of up to 4096 blocks take the one-launch cluster form (the Top-k
    in the leader CTA, 4096 being the longest row it holds); 4097 and 16384
    the two-grid form. Both run the same CTA-wide Top-k core."""
    rng = np.random.default_rng(42 + max_blocks)
    rows = _rows(rng, max_blocks)
    batch, Hkv, d, B = len(rows), 1, 64, 16
    k_max = max_blocks
    dev = torch.device("cuda:0")
    p = K.problem(batch, 1, Hkv, d, B, max_blocks, k_max)
    form, _ = K.kvsel_score_path_for(p)
    assert form == (K.KVSEL_SCORE_PATH_CLUSTER if max_blocks <= 4096 else K.KVSEL_SCORE_PATH_TWO_GRID)
    summ = torch.zeros((batch, max_blocks, Hkv, d), dtype=torch.bfloat16)
    want_vals = []
    for b, (v, _) in enumerate(rows):
        vb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
        neg_nan = np.signbit(v) & np.isnan(v)
        if neg_nan.any():                     # keep the sign bit of a negative NaN
            vb.view(torch.int16)[torch.from_numpy(neg_nan)] = torch.tensor(-64, dtype=torch.int16)  # 0xFFC0
        summ[b, : len(v), 0, 0] = vb
        want_vals.append(vb.float().numpy().astype(np.float64))
    q = torch.zeros((batch, 1, d), dtype=torch.bfloat16)
    q[:, 0, 0] = 1.0
    lens = torch.tensor([len(v) * B for v, _ in rows], dtype=torch.int32)
    ks = torch.tensor([k for _, k in rows], dtype=torch.int32)
    sel = torch.full((batch, k_max), -1, dtype=torch.int32, device=dev)
    n_sel = torch.zeros(batch, dtype=torch.int32, device=dev)
    st = torch.zeros_like(sel); ln = torch.zeros_like(sel)
    n_sp = torch.zeros_like(n_sel)
    dense = torch.zeros(batch, dtype=torch.uint8, device=dev)
    scores = torch.zeros((batch, max_blocks), dtype=torch.float32, device=dev)
    ws = torch.zeros(K.kvsel_workspace_size(p, K.KVSEL_WS_SCORE_TOPK), dtype=torch.uint8, device=dev)
    gamma, tau = 0.6, 0.5
    for _ in range(2):                        # twice: a call leaves nothing behind that changes the next
        K.kvsel_score_topk(p, q.to(dev), summ.to(dev), lens.to(dev), ks.to(dev), sel, n_sel, st, ln, n_sp, ws,
                           gamma=gamma, tau_rel=tau, dense_flag=dense, scores_out=scores)
        torch.cuda.synchronize()
        assert K.kvsel_get_error() == 0
        for b, (v, k) in enumerate(rows):
            N = len(v)
            sc = scores[b, :N].cpu().numpy().astype(np.float64)
            assert np.array_equal(sc, want_vals[b], equal_nan=True)
            want = o.topk_blocks(want_vals[b], k)
            got = sel[b, : int(n_sel[b])].cpu().numpy()
            assert np.array_equal(got, want), f"row {b}"
            a_, l_ = o.merge_spans(want)
            ns = int(n_sp[b])
            assert ns == len(a_)
            assert np.array_equal(st[b, :ns].cpu().numpy(), a_) and np.array_equal(ln[b, :ns].cpu().numpy(), l_)
            assert bool(dense[b]) == o.dense_fallback(len(a_), len(want), N, gamma, tau)
