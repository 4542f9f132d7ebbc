"""Helpers shared by the GPU parity tests: run one layer through the C ABI and
compare against the fp64 oracle with the selection tie rule.

Tie rule: indices and spans must match the oracle bit for bit unless the
oracle's k-th and (k+1)-th scores differ by less than 1e-4 relative; then the
GPU's set must still be a valid Top-k within that margin, and attention is
compared on the GPU's set.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as o
from workloads.generate import bits, logical_kv

TIE_REL = 1e-4
ATOL_MAX = 1e-2
ATOL_MEAN = 1e-3


def selection_verdict(scores: np.ndarray, k: int, gpu_sel: np.ndarray) -> str:
    """'exact', 'tie' (valid alternative inside the tie margin) or raises."""
    N = len(scores)
    k = max(0, min(k, N))
    want = o.topk_blocks(scores, k)
    gpu_sel = np.asarray(gpu_sel, dtype=np.int64)
    if np.array_equal(want, gpu_sel):
        return "exact"
    assert len(gpu_sel) == k, f"GPU selected {len(gpu_sel)} blocks, expected {k}"
    assert np.all(np.diff(gpu_sel) > 0), "GPU selection not strictly ascending"
    srt = np.sort(scores)[::-1]
    kth, nxt = srt[k - 1], srt[k]
    scale = max(abs(kth), abs(nxt), 1e-30)
    gap = abs(kth - nxt) / scale
    assert gap < TIE_REL, f"selection differs outside the tie margin (gap {gap:.3e}): {want} vs {gpu_sel}"
    margin = TIE_REL * scale
    unsel = np.setdiff1d(np.arange(N), gpu_sel)
    assert scores[gpu_sel].min() >= kth - margin
    if len(unsel):
        assert scores[unsel].max() <= kth + margin
    return "tie"


def seq_inputs(x: dict, b: int, T: int):
    """bf16 bit arrays of sequence b: q [H_q][d], K and V [T][H_kv][d]."""
    qb = bits(x["q"][b])
    kb = bits(logical_kv(x["kv_pages"], x["block_table"], b, T, 0))
    vb = bits(logical_kv(x["kv_pages"], x["block_table"], b, T, 1))
    return qb, kb, vb


def attn_errors(gpu_out: np.ndarray, ref_out: np.ndarray):
    d = np.abs(np.asarray(gpu_out, np.float64) - ref_out)
    return float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0


def check_sequence(dec, x, b, T, B, k, scale, gamma=2.0, tau_rel=0.0, scores_gpu=None,
                   summaries_gpu=None, check_spans=True):
    """Full per-sequence check of GPU outputs held by ``dec`` against the oracle."""
    qb, kb, vb = seq_inputs(x, b, T)
    N = o.n_blocks(T, B)
    sb = None
    if T > 0:
        sb, _, _ = o.block_summaries(kb, T, B)
        if summaries_gpu is not None:
            assert np.array_equal(bits(summaries_gpu[b, :N]), sb), f"summaries differ (seq {b})"
    scores = o.block_scores(qb, sb) if N > 0 else np.zeros(0)
    if scores_gpu is not None and N > 0:
        sg = scores_gpu[b, :N].double().cpu().numpy()
        assert np.abs(sg - scores).max() <= 1e-5 * max(1.0, np.abs(scores).max()), "scores differ"
    n = int(dec.n_sel[b])
    gsel = dec.sel_idx[b, :n].cpu().numpy().astype(np.int64)
    verdict = selection_verdict(scores, k, gsel)
    if check_spans:
        st, ln = o.merge_spans(gsel)
        ns = int(dec.n_spans[b])
        assert ns == len(st)
        assert np.array_equal(dec.span_start[b, :ns].cpu().numpy(), st)
        assert np.array_equal(dec.span_len[b, :ns].cpu().numpy(), ln)
    dense = N > 0 and o.dense_fallback(len(o.merge_spans(gsel)[0]), len(gsel), N, gamma, tau_rel)
    assert bool(dec.dense_flag[b]) == dense, f"dense flag differs (seq {b})"
    blocks = np.arange(N) if dense else gsel
    ref_out, ref_lse = o.attend(qb, kb, vb, o.tokens_of_blocks(blocks, T, B), scale)
    out = dec.out[b].double().cpu().numpy()
    lse = dec.lse[b].double().cpu().numpy()
    emax, emean = attn_errors(out, ref_out)
    assert emax <= ATOL_MAX and emean <= ATOL_MEAN, (b, emax, emean)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-3 * max(1.0, np.abs(ref_lse[fin]).max())
    return verdict, emax, emean


def device():
    return torch.device("cuda:0")


def to_dev(x: dict, dev) -> dict:
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in x.items()}


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
