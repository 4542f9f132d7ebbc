"""Pins of the fp64 oracle to facts fixed outside the oracle itself.

Each test ties one oracle function to something independent of it: a worked
number printed on the pages (tests/golden), a closed form, an invariant, a
library routine (torch SDPA, logsumexp, torch's fp32->bf16 conversion), exact
rational arithmetic, or brute force on tiny inputs.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as o
from workloads import C0, C1
from workloads.generate import bits, generate_layer, logical_kv

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _rows(path):
    with open(path) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- KV bytes ---

def test_kv_bytes_per_token_worked_examples(golden_dir):
    rows = _rows(os.path.join(golden_dir, "kv_bytes_worked_examples.txt"))
    per_token = {}
    for r in rows:
        if r.startswith("@total"):
            _, tokens, batch, total = r.split()
            assert o.kv_bytes_per_token(32, 2, 128, 2) * int(tokens) * int(batch) == int(total)
        elif r.startswith("@ratio"):
            assert o.kv_bytes_per_token(40, 40, 128, 2) // o.kv_bytes_per_token(32, 2, 128, 2) == int(r.split()[1])
            assert o.kv_bytes_per_token(40, 40, 128, 2) % o.kv_bytes_per_token(32, 2, 128, 2) == 0
        else:
            L, H, d, e, want = map(int, r.split())
            assert o.kv_bytes_per_token(L, H, d, e) == want
            per_token[(L, H)] = want
    assert per_token[(32, 2)] == 32 * 1024            # "32 KiB"
    assert per_token[(40, 40)] == 800 * 1024          # "800 KB"


def _round_sig(x, sig):
    return float(f"{x:.{sig}g}")


def test_transfer_time_worked_example(golden_dir):
    rows = _rows(os.path.join(golden_dir, "transfer_time_worked_example.txt"))
    times = []
    for r in rows:
        if r.startswith("@ratio_about"):
            ratio = times[1] / times[0]
            assert abs(ratio - float(r.split()[1])) / float(r.split()[1]) < 0.1
            continue
        nbytes, bw, ms, sig = r.split()
        t = o.transfer_seconds(float(nbytes), float(bw))
        times.append(t)
        assert _round_sig(t * 1e3, int(sig)) == float(ms)


# ------------------------------------------------------------- bf16 RNE ---

def _all_finite_positive_bf16():
    b = np.arange(0, 0x7F80, dtype=np.uint16)      # +0 .. largest finite
    return b, o.bf16_bits_to_f64(b)


def test_rne_identity_on_every_bf16_value():
    b = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    v = o.bf16_bits_to_f64(b)
    r = o.rne_bf16_bits(v)
    fin = ~np.isnan(v)
    assert np.array_equal(r[fin], b[fin])
    assert np.all((r[~fin] & 0x7FFF) == 0x7FC0)


def test_rne_midpoints_go_to_even_and_neighbours_to_nearest():
    b, v = _all_finite_positive_bf16()
    lo, hi = v[:-1], v[1:]
    mid = (lo + hi) / 2                      # exact in fp64 (bf16 has 8 bits)
    r = o.rne_bf16_bits(mid)
    even = np.where((b[:-1] & 1) == 0, b[:-1], b[1:])
    assert np.array_equal(r, even)
    below = np.nextafter(mid, -np.inf)
    above = np.nextafter(mid, np.inf)
    assert np.array_equal(o.rne_bf16_bits(below), b[:-1])
    assert np.array_equal(o.rne_bf16_bits(above), b[1:])
    assert np.array_equal(o.rne_bf16_bits(-above), b[1:] | 0x8000)
    top = v[-1]
    half_ulp = (top - v[-2]) / 2
    assert o.rne_bf16_bits(np.array([top + half_ulp]))[0] == 0x7F80     # tie -> even = inf
    assert o.rne_bf16_bits(np.array([np.nextafter(top + half_ulp, 0)]))[0] == 0x7F7F
    assert o.rne_bf16_bits(np.array([-0.0]))[0] == 0x8000


def test_rne_matches_library_on_fp32_inputs():
    g = np.random.default_rng(5)
    x32 = np.concatenate([
        g.standard_normal(200000).astype(np.float32),
        (g.standard_normal(20000) * 1e-39).astype(np.float32),     # fp32 subnormals
        (g.standard_normal(20000) * 3e37).astype(np.float32),
    ])
    lib = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = o.rne_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(mine, lib)


# ------------------------------------------------------------- summaries ---

_POS_GRID = None


def _rne_fraction(q: Fraction) -> int:
    """Exact round-to-nearest-even of a rational to bf16 by bisection on the grid."""
    global _POS_GRID
    if _POS_GRID is None:
        _POS_GRID = [Fraction(float(x)) for x in o.bf16_bits_to_f64(np.arange(0, 0x7F80, dtype=np.uint16))]
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    lo, hi = 0, len(_POS_GRID) - 1
    while hi - lo > 1:
        m = (lo + hi) // 2
        if _POS_GRID[m] <= a:
            lo = m
        else:
            hi = m
    if a >= _POS_GRID[hi]:
        lo = hi
    if lo == len(_POS_GRID) - 1 or a == _POS_GRID[lo]:
        r = lo
    else:
        dl, dh = a - _POS_GRID[lo], _POS_GRID[lo + 1] - a
        r = lo if dl < dh else lo + 1 if dh < dl else (lo if lo % 2 == 0 else lo + 1)
    return r | sign if (r or sign == 0) else sign


def test_summaries_equal_exact_rational_mean_rounded_once():
    g = np.random.default_rng(11)
    T, B, H, d = 13, 4, 2, 8                        # 4 blocks, the last one partial
    kb = o.rne_bf16_bits(g.standard_normal((T, H, d)) * 3.0)
    sbits, means, last = o.block_summaries(kb, T, B)
    kf = o.bf16_bits_to_f64(kb)
    N = o.n_blocks(T, B)
    assert sbits.shape == (N, H, d)
    for n in range(N):
        toks = range(n * B, min(T, n * B + B))
        for j in range(H):
            for c in range(d):
                exact = sum(Fraction(float(kf[t, j, c])) for t in toks) / len(toks)
                assert sbits[n, j, c] == _rne_fraction(exact), (n, j, c)


def test_summary_closed_forms():
    B, H, d = 8, 2, 4
    T = 3 * B + 3
    const = np.full((T, H, d), 0.3)
    kb = o.rne_bf16_bits(const)
    s, _, _ = o.block_summaries(kb, T, B)
    assert np.all(s == kb[0, 0, 0])                       # constant block -> constant
    pm = np.empty((4 * B, H, d))
    pm[0::2] = 1.75
    pm[1::2] = -1.75
    s, _, _ = o.block_summaries(o.rne_bf16_bits(pm), 4 * B, B)
    assert np.all(o.bf16_bits_to_f64(s) == 0.0)          # +-x pairs -> 0
    one = o.rne_bf16_bits(np.random.default_rng(1).standard_normal((5, H, d)))
    s, _, _ = o.block_summaries(one, 5, 1)
    assert np.array_equal(s, one)                         # one-token blocks -> the key


def test_incremental_append_equals_rebuild():
    g = np.random.default_rng(3)
    B, H, d = 16, 2, 8
    T0, T1 = 37, 70
    kb = o.rne_bf16_bits(g.standard_normal((T1, H, d)))
    _, _, acc = o.block_summaries(kb, T0, B)
    for t in range(T0, T1):
        acc, sb = o.append_token(acc, kb[t], t, B)
        full, _, last = o.block_summaries(kb, t + 1, B)
        assert np.array_equal(sb, full[t // B])
        assert np.array_equal(acc, last)


# ------------------------------------------------------------------ score ---

def test_score_linearity_over_tokens():
    """sum_h q_h . mean(K) == mean over tokens of sum_h q_h . k_t (unrounded means)."""
    g = np.random.default_rng(7)
    T, B, Hq, Hkv, d = 96, 16, 8, 2, 32
    kb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    qb = o.rne_bf16_bits(g.standard_normal((Hq, d)))
    _, means, _ = o.block_summaries(kb, T, B)
    score = o.block_scores(qb, means, summary_is_bits=False)
    q = o.bf16_bits_to_f64(qb)
    K = o.bf16_bits_to_f64(kb)
    G = Hq // Hkv
    per_token = np.array([sum(q[h] @ K[t, h // G] for h in range(Hq)) for t in range(T)])
    want = per_token.reshape(-1, B).mean(axis=1)
    assert np.allclose(score, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_score_gqa_equals_mha_with_replicated_kv_heads():
    g = np.random.default_rng(8)
    N, Hq, Hkv, d = 12, 8, 2, 16
    s = o.rne_bf16_bits(g.standard_normal((N, Hkv, d)))
    qb = o.rne_bf16_bits(g.standard_normal((Hq, d)))
    s_mha = np.repeat(s, Hq // Hkv, axis=1)           # head h reads KV head h // G
    assert np.array_equal(o.block_scores(qb, s), o.block_scores(qb, s_mha))


def test_score_one_hot_query_reads_one_summary_entry():
    g = np.random.default_rng(9)
    N, Hq, Hkv, d = 10, 6, 3, 8
    s = o.rne_bf16_bits(g.standard_normal((N, Hkv, d)))
    sf = o.bf16_bits_to_f64(s)
    for h, c in [(0, 0), (1, 5), (4, 7), (5, 2)]:
        q = np.zeros((Hq, d))
        q[h, c] = 1.0
        assert np.array_equal(o.block_scores(o.rne_bf16_bits(q), s), sf[:, h // 2, c])


# ------------------------------------------------------------------ top-k ---

def _brute_topk(scores, k):
    N = len(scores)
    best = None
    for sub in itertools.combinations(range(N), k):
        rest = [i for i in range(N) if i not in sub]
        if rest and min(scores[i] for i in sub) < max(scores[i] for i in rest):
            continue
        # among valid sets, ties go to lower indices: the lexicographically
        # smallest set after sorting by (score desc, index asc)
        key = sorted(sub, key=lambda i: (-scores[i], i))
        if best is None or [(-scores[i], i) for i in key] < [(-scores[i], i) for i in best]:
            best = key
    return sorted(best)


@pytest.mark.parametrize("seed", range(40))
def test_topk_brute_force_with_ties(seed):
    g = np.random.default_rng(seed)
    N = int(g.integers(1, 9))
    scores = g.integers(-2, 3, size=N).astype(np.float64)    # many exact ties
    for k in range(0, N + 1):
        got = o.topk_blocks(scores, k).tolist()
        want = _brute_topk(list(scores), k) if k else []
        assert got == want, (scores, k)


def test_topk_ranks_nan_below_every_number():
    # worked by hand: 2 (block 4), 1 (block 1), -inf (block 2), then the NaNs
    # by index (blocks 0 and 3)
    s = np.array([np.nan, 1.0, -np.inf, np.nan, 2.0])
    want = {1: [4], 2: [1, 4], 3: [1, 2, 4], 4: [0, 1, 2, 4], 5: [0, 1, 2, 3, 4]}
    for k, sel in want.items():
        assert o.topk_blocks(s, k).tolist() == sel


def test_topk_clamps_k():
    s = np.array([3.0, 1.0, 2.0])
    assert o.topk_blocks(s, 7).tolist() == [0, 1, 2]
    assert o.topk_blocks(s, -1).tolist() == []
    assert o.topk_blocks(np.zeros(0), 4).tolist() == []


def _brute_window(scores, k, n_sink, n_recent):
    """Every block set that holds the forced blocks and min(k, #candidates)
    others, keeping the sets whose added blocks all score at least as high as
    every candidate left out; among those the lowest indices win ties."""
    N = len(scores)
    forced = {i for i in range(N) if i < n_sink or i >= N - n_recent}
    cands = [i for i in range(N) if i not in forced]
    kk = max(0, min(k, len(cands)))
    best = None
    for sub in itertools.combinations(range(N), len(forced) + kk):
        if not forced <= set(sub):
            continue
        added = [i for i in sub if i not in forced]
        left = [i for i in cands if i not in sub]
        if added and left and min(scores[i] for i in added) < max(scores[i] for i in left):
            continue
        key = sorted(added, key=lambda i: (-scores[i], i))
        if best is None or [(-scores[i], i) for i in key] < [(-scores[i], i) for i in best[0]]:
            best = (key, sorted(sub))
    return best[1]


@pytest.mark.parametrize("seed", range(30))
def test_window_select_brute_force_with_ties(seed):
    g = np.random.default_rng(100 + seed)
    N = int(g.integers(0, 9))
    scores = g.integers(-2, 3, size=N).astype(np.float64)
    for n_sink in range(0, 3):
        for n_recent in range(0, 4):
            for k in range(0, N + 1):
                got = o.window_select(scores, k, n_sink, n_recent).tolist()
                assert got == _brute_window(list(scores), k, n_sink, n_recent), (scores, k, n_sink, n_recent)


def test_zero_window_is_plain_topk():
    g = np.random.default_rng(7)
    for _ in range(50):
        sc = g.standard_normal(int(g.integers(1, 40)))
        k = int(g.integers(0, len(sc) + 1))
        assert np.array_equal(o.window_select(sc, k, 0, 0), o.topk_blocks(sc, k))


# ------------------------------------------------------------------ spans ---

def test_spans_hand_examples(golden_dir):
    for r in _rows(os.path.join(golden_dir, "spans_hand_example.txt")):
        sel, st, ln = (list(map(int, p.split())) for p in r.split("|"))
        a, b = o.merge_spans(np.array(sel))
        assert a.tolist() == st and b.tolist() == ln


def test_span_invariants():
    g = np.random.default_rng(2)
    for _ in range(200):
        N = int(g.integers(1, 60))
        k = int(g.integers(0, N + 1))
        sel = np.sort(g.choice(N, size=k, replace=False))
        st, ln = o.merge_spans(sel)
        assert ln.sum() == k
        rebuilt = np.concatenate([np.arange(s, s + l) for s, l in zip(st, ln)]) if k else np.zeros(0)
        assert np.array_equal(rebuilt, sel)
        assert np.all(st[1:] >= st[:-1] + ln[:-1] + 1)    # disjoint, sorted, gap >= 1


# -------------------------------------------------------------- attention ---

def _sdpa_full(qb, kb, vb, T, scale):
    q = torch.from_numpy(o.bf16_bits_to_f64(qb))[None, :, None, :]
    K = torch.from_numpy(o.bf16_bits_to_f64(kb[:T])).permute(1, 0, 2)[None]
    V = torch.from_numpy(o.bf16_bits_to_f64(vb[:T])).permute(1, 0, 2)[None]
    G = q.shape[1] // K.shape[1]
    K = K.repeat_interleave(G, dim=1)
    V = V.repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)
    lse = torch.logsumexp((q @ K.transpose(-1, -2)) * scale, dim=-1)
    return out[0, :, 0].numpy(), lse[0, :, 0].numpy()


@pytest.mark.parametrize("Hq,Hkv,T,B", [(8, 8, 200, 16), (8, 2, 131, 32), (4, 1, 64, 64)])
def test_k_equal_n_and_gamma_dense_equal_full_attention(Hq, Hkv, T, B):
    g = np.random.default_rng(T)
    d = 32
    qb = o.rne_bf16_bits(g.standard_normal((Hq, d)))
    kb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    vb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    scale = 1.0 / math.sqrt(d)
    want, want_lse = _sdpa_full(qb, kb, vb, T, scale)
    N = o.n_blocks(T, B)
    r = o.decode_seq(qb, kb, vb, T, B, N, scale)                # k = N
    assert not r.dense and len(r.sel) == N
    assert np.allclose(r.out, want, atol=1e-12, rtol=1e-10)
    assert np.allclose(r.lse, want_lse, atol=1e-12, rtol=1e-12)
    r = o.decode_seq(qb, kb, vb, T, B, 1, scale, gamma=0.0)     # gamma forces dense
    assert r.dense and len(r.sel) == 1
    assert np.allclose(r.out, want, atol=1e-12, rtol=1e-10)


def test_sparse_attention_equals_masked_library_attention():
    g = np.random.default_rng(21)
    Hq, Hkv, T, B, d = 8, 4, 150, 16, 32
    qb = o.rne_bf16_bits(g.standard_normal((Hq, d)))
    kb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    vb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    scale = 0.17
    r = o.decode_seq(qb, kb, vb, T, B, 4, scale)
    mask = np.zeros(T, dtype=bool)
    for s in r.sel:
        mask[s * B: min(T, s * B + B)] = True
    q = torch.from_numpy(o.bf16_bits_to_f64(qb))[None, :, None, :]
    K = torch.from_numpy(o.bf16_bits_to_f64(kb)).permute(1, 0, 2)[None].repeat_interleave(2, dim=1)
    V = torch.from_numpy(o.bf16_bits_to_f64(vb)).permute(1, 0, 2)[None].repeat_interleave(2, dim=1)
    want = torch.nn.functional.scaled_dot_product_attention(
        q, K, V, attn_mask=torch.from_numpy(mask)[None, None, None, :], scale=scale)[0, :, 0].numpy()
    assert np.allclose(r.out, want, atol=1e-12, rtol=1e-10)


def test_window_halves_merged_by_lse_equal_one_attention_over_the_union():
    # [DKV]: the recency window is attended exactly, the Top-k blocks apart,
    # and the two halves are merged by the log-sum-exp reduction. That merge
    # must equal one softmax over the union of their tokens, which is what the
    # oracle computes; both also match masked library attention.
    g = np.random.default_rng(33)
    Hq, Hkv, T, B, d = 8, 2, 300, 16, 32
    qb = o.rne_bf16_bits(g.standard_normal((Hq, d)))
    kb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    vb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    scale = 0.21
    n_sink, n_recent, k = 1, 3, 4
    r = o.decode_seq(qb, kb, vb, T, B, k, scale, n_sink=n_sink, n_recent=n_recent)
    N = o.n_blocks(T, B)
    window = [n for n in r.sel if n < n_sink or n >= N - n_recent]
    topk = [n for n in r.sel if n_sink <= n < N - n_recent]
    assert window == [0, N - 3, N - 2, N - 1] and len(topk) == k
    o1, l1 = o.attend(qb, kb, vb, o.tokens_of_blocks(window, T, B), scale)
    o2, l2 = o.attend(qb, kb, vb, o.tokens_of_blocks(topk, T, B), scale)
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    merged = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None]
    assert np.allclose(r.out, merged, atol=1e-13, rtol=1e-11)
    assert np.allclose(r.lse, m + np.log(w1 + w2), atol=1e-13, rtol=1e-13)
    mask = np.zeros(T, dtype=bool)
    for s in r.sel:
        mask[s * B: min(T, s * B + B)] = True
    q = torch.from_numpy(o.bf16_bits_to_f64(qb))[None, :, None, :]
    K = torch.from_numpy(o.bf16_bits_to_f64(kb)).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    V = torch.from_numpy(o.bf16_bits_to_f64(vb)).permute(1, 0, 2)[None].repeat_interleave(4, dim=1)
    want = torch.nn.functional.scaled_dot_product_attention(
        q, K, V, attn_mask=torch.from_numpy(mask)[None, None, None, :], scale=scale)[0, :, 0].numpy()
    assert np.allclose(r.out, want, atol=1e-12, rtol=1e-10)


def test_window_covering_every_block_is_full_attention():
    g = np.random.default_rng(34)
    Hq, Hkv, T, B, d = 4, 2, 170, 32, 16
    qb = o.rne_bf16_bits(g.standard_normal((Hq, d)))
    kb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    vb = o.rne_bf16_bits(g.standard_normal((T, Hkv, d)))
    want, want_lse = _sdpa_full(qb, kb, vb, T, 0.3)
    N = o.n_blocks(T, B)
    for n_sink, n_recent in ((0, N), (N, 0), (2, N - 2), (3, 9)):
        r = o.decode_seq(qb, kb, vb, T, B, 1, 0.3, n_sink=n_sink, n_recent=n_recent)
        assert r.sel.tolist() == list(range(N))
        assert np.allclose(r.out, want, atol=1e-12, rtol=1e-10)
        assert np.allclose(r.lse, want_lse, atol=1e-12, rtol=1e-12)


def test_attention_closed_forms():
    g = np.random.default_rng(4)
    Hq, Hkv, d = 4, 2, 16
    qb = o.rne_bf16_bits(g.standard_normal((Hq, d)))
    vb = o.rne_bf16_bits(g.standard_normal((40, Hkv, d)))
    kb = o.rne_bf16_bits(g.standard_normal((40, Hkv, d)))
    out, lse = o.attend(qb, kb, vb, np.array([17]), 0.25)       # one token -> o = v
    V = o.bf16_bits_to_f64(vb)
    for h in range(Hq):
        assert np.array_equal(out[h], V[17, h // 2])
    kc = np.broadcast_to(kb[:1], kb.shape).copy()               # constant keys -> mean(V)
    toks = np.arange(3, 29)
    out, _ = o.attend(qb, kc, vb, toks, 0.25)
    for h in range(Hq):
        assert np.allclose(out[h], V[toks, h // 2].mean(axis=0), atol=1e-14)
    out, lse = o.attend(qb, kb, vb, np.zeros(0, dtype=np.int64), 0.25)   # empty set
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_empty_sequence():
    qb = o.rne_bf16_bits(np.ones((2, 8)))
    kb = np.zeros((0, 1, 8), dtype=np.uint16)
    r = o.decode_seq(qb, kb, kb, 0, 16, 4, 0.3)
    assert len(r.sel) == 0 and len(r.span_start) == 0 and not r.dense
    assert np.all(r.out == 0) and np.all(np.isneginf(r.lse))


# ----------------------------------------------------------------- budget ---

def test_budget_hand_examples(golden_dir):
    for r in _rows(os.path.join(golden_dir, "budget_hand_examples.txt")):
        lhs, rhs = r.split("|")
        B, H, d, e, hid, N = map(int, lhs.split()[:6])
        bw, F, kappa, floor, gamma, tau, ovr = map(float, lhs.split()[6:])
        c_copy, c_rec, r_model, rr, k, dense = rhs.split()
        out = o.budget(B, H, d, e, hid, N, bw, F, kappa, floor, gamma, tau, ovr)
        assert out.c_copy_s == float(c_copy)
        assert out.c_rec_s == float(c_rec)
        assert out.r_model == float(r_model)
        assert out.r == float(rr)
        assert out.k == int(k)
        assert out.dense == bool(int(dense))


def test_dense_rule_boundaries():
    assert o.dense_fallback(1, 8, 10, 0.8, 0.0)           # k == gamma*N -> dense
    assert not o.dense_fallback(1, 7, 10, 0.8, 0.0)
    assert o.dense_fallback(1, 10, 10, 1.0, 0.0)          # k == N, gamma = 1 -> dense
    assert not o.dense_fallback(1, 10, 10, 1.01, 0.0)
    assert o.dense_fallback(3, 7, 10, 0.8, 1.0)           # 3 + 7 >= 8.8
    assert not o.dense_fallback(1, 7, 10, 0.8, 1.0)       # 1 + 7 <  8.8


# ---------------------------------------------------------------- needles ---

@pytest.mark.parametrize("layer", [0, 1])
def test_planted_needles_are_selected_at_both_keep_ratios(layer):
    w = C1
    x = generate_layer(w, layer)
    B = w.block_size
    for b in range(w.batch):
        kb = bits(logical_kv(x["kv_pages"], x["block_table"], b, w.seq_len, 0))
        s, _, _ = o.block_summaries(kb, w.seq_len, B)
        sc = o.block_scores(bits(x["q"][b]), s)
        for k in w.ks:
            sel = set(o.topk_blocks(sc, k).tolist())
            assert set(w.needles) <= sel, (b, k)
        # the needle margin is huge: about 4*sum_h |q_h|^2 against noise ~ 16
        order = np.sort(sc)[::-1]
        assert order[1] > 50 * np.abs(np.delete(sc, list(w.needles))).max() / 10


def test_c0_step_runs_and_is_self_consistent():
    w = C0
    x = generate_layer(w)
    kb = bits(logical_kv(x["kv_pages"], x["block_table"], 0, w.seq_len, 0))
    vb = bits(logical_kv(x["kv_pages"], x["block_table"], 0, w.seq_len, 1))
    r = o.decode_seq(bits(x["q"][0]), kb, vb, w.seq_len, w.block_size, w.topk, 1 / 8)
    assert len(r.sel) == w.topk and r.span_len.sum() == w.topk
    assert np.all(np.isfinite(r.out)) and np.all(np.isfinite(r.lse))


# ------------------------------------------------------------ block cache ---

def _replay_cache_example(cls, path, slots):
    """Replays a hand-worked cache example (step rows and prefetch rows 'P');
    returns the first row whose outcome differs, or None."""
    c = cls(slots)
    for r in _rows(path):
        kind, blocks, last, jobs, hits, blk, use = (p.strip() for p in r.split("|"))
        blocks = [int(v) for v in blocks.split()]
        if kind == "P":
            got_jobs, got_hits = c.prefetch(blocks, int(last)), []
        else:
            got_jobs, got_hits = c.step(blocks, int(kind), int(last))
        want_jobs = [] if jobs == "-" else [tuple(int(x) for x in j.split(":")) for j in jobs.split()]
        if (got_jobs != want_jobs or got_hits != ([] if hits == "-" else [int(v) for v in hits.split()])
                or c.block_in != [int(v) for v in blk.split()] or c.last_use != [int(v) for v in use.split()]):
            return r
    return None


def test_block_cache_hand_example(golden_dir):
    assert _replay_cache_example(o.BlockCache, os.path.join(golden_dir, "block_cache_hand_example.txt"), 3) is None


def test_block_cache_prefetch_hand_example(golden_dir):
    path = os.path.join(golden_dir, "block_cache_prefetch_hand_example.txt")
    assert _replay_cache_example(o.BlockCache, path, 4) is None


# Plausible mistakes in the cache, each planted in a copy of the oracle's
# class; the hand-worked examples must catch every one of them.
class _MruOrder(o.BlockCache):
    def step(self, sel, step, last_block):
        save = list(self.last_use)
        self.last_use = [-2 - u if u >= 0 else u for u in save]   # newest first among used slots
        try:
            jobs, hits = super().step(sel, step, last_block)
        finally:
            self.last_use = [step if u == step else (-2 - u if u <= -2 else u) for u in self.last_use]
        return jobs, hits


class _ReversedSlotTies(o.BlockCache):
    def step(self, sel, step, last_block):
        self.block_in.reverse(); self.last_use.reverse()
        self.slot_of = {b: self.slots - 1 - s for b, s in self.slot_of.items()}
        jobs, hits = super().step(sel, step, last_block)
        self.block_in.reverse(); self.last_use.reverse()
        self.slot_of = {b: self.slots - 1 - s for b, s in self.slot_of.items()}
        return [(n, self.slots - 1 - s) for n, s in jobs], hits


class _NoRefresh(o.BlockCache):
    def step(self, sel, step, last_block):
        return super().step(sel, step, -1)


class _ReversedMissOrder(o.BlockCache):
    def step(self, sel, step, last_block):
        jobs, hits = super().step(sel, step, last_block)
        n_miss = len([j for j in jobs if j[0] not in hits])
        misses = jobs[:n_miss]
        blocks = [n for n, _ in misses][::-1]
        for (n, s), m in zip(misses, blocks):
            self.block_in[s] = m
            self.slot_of[m] = s
        return [(m, s) for (_, s), m in zip(misses, blocks)] + jobs[n_miss:], hits


class _PrefetchStamped(o.BlockCache):
    def prefetch(self, pred, last_block):
        jobs = super().prefetch(pred, last_block)
        top = max(self.last_use)
        for _, s in jobs:
            self.last_use[s] = top                  # as if selected in the last step
        return jobs


class _PrefetchEvictsPredicted(o.BlockCache):
    def prefetch(self, pred, last_block):
        keep = dict(self.slot_of)
        self.slot_of = {}                           # forget which slots hold predicted blocks
        misses = [n for n in pred if n not in keep and n != last_block]
        free = sorted(range(self.slots), key=lambda s: (self.last_use[s], s))
        self.slot_of = keep
        jobs = []
        for n, s in zip(misses, free):
            old = self.block_in[s]
            if old >= 0:
                del self.slot_of[old]
            self.block_in[s], self.slot_of[n], self.last_use[s] = n, s, -1
            jobs.append((n, s))
        return jobs


class _PrefetchTakesLastBlock(o.BlockCache):
    def prefetch(self, pred, last_block):
        return super().prefetch(pred, -1)


class _PrefetchTouchesResident(o.BlockCache):
    def prefetch(self, pred, last_block):
        jobs = super().prefetch(pred, last_block)
        for n in pred:
            s = self.slot_of.get(n)
            if s is not None and self.last_use[s] >= 0:
                self.last_use[s] += 1
        return jobs


@pytest.mark.parametrize("mutant", [_MruOrder, _ReversedSlotTies, _NoRefresh, _ReversedMissOrder,
                                    _PrefetchStamped, _PrefetchEvictsPredicted,
                                    _PrefetchTakesLastBlock, _PrefetchTouchesResident])
def test_block_cache_examples_catch_planted_mistakes(golden_dir, mutant):
    caught = [_replay_cache_example(mutant, os.path.join(golden_dir, name), slots) is not None
              for name, slots in (("block_cache_hand_example.txt", 3),
                                  ("block_cache_prefetch_hand_example.txt", 4))]
    assert any(caught), mutant.__name__


def _random_selections(g, steps, N, k, locality):
    sel = np.sort(g.choice(N, size=k, replace=False))
    out = []
    for _ in range(steps):
        keep = sel[g.random(k) < locality]
        rest = np.setdiff1d(np.arange(N), keep)
        sel = np.sort(np.concatenate([keep, g.choice(rest, size=k - len(keep), replace=False)]))
        out.append(sel)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_block_cache_invariants_and_lru_order_from_history(seed):
    g = np.random.default_rng(seed)
    N, k = 40, int(g.integers(3, 9))
    slots = k + int(g.integers(0, 7))
    c = o.BlockCache(slots)
    last_sel = {}                       # block -> last step it was selected (raw history)
    resident_prev = set()
    for step, sel in enumerate(_random_selections(g, 60, N, k, 0.7)):
        last = int(g.integers(N - 3, N))
        jobs, hits = c.step(sel, step, last)
        sel_set = set(sel.tolist())
        resident = {b for b in c.block_in if b >= 0}
        # every selected block is resident; hits were resident before
        assert sel_set <= resident and set(hits) <= resident_prev
        assert len(resident) <= slots
        # block_in and slot_of are inverse maps
        assert all(c.block_in[s] == b for b, s in c.slot_of.items())
        assert len(c.slot_of) == len(resident)
        misses = sorted(sel_set - set(hits))
        assert [n for n, _ in jobs[:len(misses)]] == misses
        assert jobs[len(misses):] == ([(last, c.slot_of[last])] if last in hits else [])
        # LRU from the raw history: no evicted block was selected later than a
        # block that stayed without being selected in this step
        evicted = resident_prev - resident
        kept_idle = (resident & resident_prev) - sel_set
        if evicted and kept_idle:
            assert max(last_sel[b] for b in evicted) <= min(last_sel[b] for b in kept_idle)
        for b in sel_set:
            last_sel[b] = step
        resident_prev = resident


@pytest.mark.parametrize("seed", range(6))
def test_block_cache_prefetch_invariants(seed):
    g = np.random.default_rng(100 + seed)
    N, k = 40, int(g.integers(3, 9))
    slots = 2 * k + int(g.integers(0, 4))
    c = o.BlockCache(slots)
    prev = np.array([], dtype=np.int64)
    for step, sel in enumerate(_random_selections(g, 60, N, k, 0.7)):
        last = int(g.integers(N - 3, N))
        # a prediction: most of the previous selection plus a few other blocks
        extra = g.choice(N, size=int(g.integers(0, k + 1)), replace=False)
        pred = np.union1d(prev[g.random(len(prev)) < 0.8], extra)[:slots]
        pred = [int(n) for n in pred]
        slot_before = dict(c.slot_of)
        use_before = list(c.last_use)
        jobs = c.prefetch(pred, last)
        resident = {b for b in c.block_in if b >= 0}
        assert all(c.block_in[s] == b for b, s in c.slot_of.items()) and len(c.slot_of) == len(resident)
        # every predicted block is resident, except a last block that was not
        assert set(pred) - {last} <= resident
        if last not in slot_before:
            assert last not in resident      # never brought in by a prefetch
        # resident predicted blocks stay where they were, stamps unchanged
        for n in pred:
            if n in slot_before:
                assert c.slot_of[n] == slot_before[n] and c.last_use[slot_before[n]] == use_before[slot_before[n]]
        # jobs: the other predicted blocks, ascending, stamped -1
        assert [n for n, _ in jobs] == sorted(n for n in pred if n not in slot_before and n != last)
        assert all(c.block_in[s] == n and c.last_use[s] == -1 for n, s in jobs)
        # victims hold no predicted block and come first in (stamp, slot) order
        evicted = set(slot_before) - resident
        assert not evicted & set(pred)
        kept_other = (set(slot_before) & resident) - set(pred)
        order = lambda b: (use_before[slot_before[b]], slot_before[b])
        if evicted and kept_other:
            assert max(map(order, evicted)) < min(map(order, kept_other))
        # the step then hits every selected block the cache now holds
        held = dict(c.slot_of)
        jobs2, hits = c.step(sel, step, last)
        assert set(hits) == {int(n) for n in sel if int(n) in held}
        prev = sel


def test_block_cache_prefetch_special_cases():
    # prefetching exactly the next selection leaves that step nothing to fetch
    # but the block holding the last token
    c = o.BlockCache(6)
    c.step([0, 1, 2], 0, 9)
    assert c.prefetch([1, 4, 5, 9], 9) == [(4, 3), (5, 4)]
    jobs, hits = c.step([1, 4, 5, 9], 1, 9)
    assert jobs == [(9, 5)] and hits == [1, 4, 5]
    # a prediction already resident fetches nothing and changes nothing
    state = (list(c.block_in), list(c.last_use))
    assert c.prefetch([1, 4, 9], 9) == [] and (c.block_in, c.last_use) == state
    assert c.prefetch([], 9) == [] and (c.block_in, c.last_use) == state
    # a wrong prediction is evicted before any block that was ever selected
    c = o.BlockCache(4)
    c.step([0, 1], 0, 50)
    assert c.prefetch([7], 50) == [(7, 2)]
    c.step([0, 1], 1, 50)
    jobs, _ = c.step([2, 3], 2, 50)
    assert jobs == [(2, 2), (3, 3)] and 7 not in c.slot_of and {0, 1} <= set(c.slot_of)


def test_block_cache_special_cases():
    # the same selection again: nothing to fetch but the refreshed last block
    c = o.BlockCache(8)
    assert len(c.step([1, 3, 9], 0, 9)[0]) == 3
    assert c.step([1, 3, 9], 1, 9) == ([(9, c.slot_of[9])], [1, 3, 9])
    assert c.step([1, 3, 9], 2, 12) == ([], [1, 3, 9])
    # disjoint selections with slots == k: every block is fetched and the
    # evicted ones are exactly the previous step's
    c = o.BlockCache(4)
    prev = None
    for step in range(5):
        sel = list(range(4 * step, 4 * step + 4))
        jobs, hits = c.step(sel, step, 100)
        assert hits == [] and [n for n, _ in jobs] == sel
        assert sorted(b for b in c.block_in) == sel
        if prev is not None:
            assert not set(prev) & set(c.block_in)
        prev = sel
