"""GPU: kvsel_append_score_topk (the token's summary append folded into the
score grid) against the two calls it replaces, kvsel_build_summaries(APPEND)
then kvsel_score_topk, bit for bit on every output, and against the fp64
oracle at the end of a run of decode steps."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests._parity import check_sequence, to_dev
from workloads import C0, C1, C3
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


@pytest.fixture(autouse=True)
def _no_device_error(K):
    K.kvsel_get_error()
    yield
    assert K.kvsel_get_error() == 0, "a kernel latched a device error"


def _decoder(w, mb, k):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, mb,
                        device="cuda:0")
    dec.k_per_seq.fill_(k)
    return dec


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


# (name, workload, starting lengths, k, decode steps). The shapes cover a
# summary row of 4 (GQA, d 128), 2 (MHA, d 64) and 16 (MHA, d 128) 16-byte
# vectors per lane, and 16 lanes per block (one KV head of d 128); the small
# tables put several sequences, and several open blocks, in one CTA's share.
CASES = [
    ("gqa8_d128_B32", C3.scaled(batch=3, seq_len=300, layers=1), [300, 257, 31], 6, 40),
    ("mha8_d64_B16", C0.scaled(batch=4, seq_len=200), [200, 190, 17, 64], 8, 40),
    ("mha32_d128_B16", C1.scaled(batch=2, seq_len=300, layers=1, needles=()), [300, 250], 10, 20),
    ("kv1_d128_B16", C0.scaled(n_qheads=4, n_kvheads=1, head_dim=128, batch=5, seq_len=150),
     [150, 3, 96, 111, 47], 5, 40),
]


@pytest.mark.parametrize("name,w,lens0,k,steps", CASES, ids=[c[0] for c in CASES])
def test_fused_append_equals_two_calls(K, name, w, lens0, k, steps):
    B = w.block_size
    mb = (max(lens0) + steps + B - 1) // B
    x = to_dev(generate_layer(w, 0, max_blocks=mb, seq_lens=lens0), "cuda:0")
    xa = dict(x, kv_pages=x["kv_pages"].clone())
    xb = dict(x, kv_pages=x["kv_pages"].clone())
    da, db = _decoder(w, mb, k), _decoder(w, mb, k)
    sa, aa = da.new_summaries()
    sb, ab = db.new_summaries()
    da.build_summaries(xa["kv_pages"], x["block_table"], x["seq_lens"], sa, aa)
    db.build_summaries(xb["kv_pages"], x["block_table"], x["seq_lens"], sb, ab)
    sc_a = torch.zeros((w.batch, mb), device="cuda:0")
    sc_b = torch.zeros((w.batch, mb), device="cuda:0")
    g = torch.Generator(device="cuda:0")
    g.manual_seed(11)
    lens = x["seq_lens"].clone()
    for step in range(steps):
        shape = (w.batch, w.n_kvheads, w.head_dim)
        new_k = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
        new_v = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
        pos = lens.clone()
        if step % 3 == 1:
            pos[step % w.batch] = -1                 # this sequence appends nothing this step
        nk, nv = (None, None) if step % 7 == 5 else (new_k, new_v)   # re-summarise the cached row
        nxt = lens + (pos >= 0).to(torch.int32)
        da.append(xa["kv_pages"], x["block_table"], pos, sa, aa, new_k=nk, new_v=nv)
        da.select(x["q"], sa, nxt, scores_out=sc_a)
        db.append_select(xb["kv_pages"], x["block_table"], pos, x["q"], sb, ab, nxt, new_k=nk,
                         new_v=nv, scores_out=sc_b)
        torch.cuda.synchronize()
        assert _same(xa["kv_pages"], xb["kv_pages"]), f"kv pages differ at step {step}"
        assert _same(sa, sb), f"summaries differ at step {step}"
        assert _same(aa, ab), f"open-block sums differ at step {step}"
        for b in range(w.batch):
            n = (int(nxt[b]) + B - 1) // B
            assert _same(sc_a[b, :n], sc_b[b, :n]), f"scores differ (seq {b}, step {step})"
        for name_ in ("n_sel", "n_spans", "dense_flag"):
            assert torch.equal(getattr(da, name_), getattr(db, name_)), (name_, step)
        for b in range(w.batch):
            ns, nsp = int(db.n_sel[b]), int(db.n_spans[b])
            assert torch.equal(da.sel_idx[b, :ns], db.sel_idx[b, :ns]), (b, step)
            assert torch.equal(da.span_start[b, :nsp], db.span_start[b, :nsp]), (b, step)
            assert torch.equal(da.span_len[b, :nsp], db.span_len[b, :nsp]), (b, step)
        lens = nxt
    # the final state against the oracle
    xb["seq_lens"] = lens
    db.attend(x["q"], K.kv_paged(xb["kv_pages"], x["block_table"]), lens)
    torch.cuda.synchronize()
    for b in range(w.batch):
        check_sequence(db, xb, b, int(lens[b]), B, k, db.scale, scores_gpu=sc_b, summaries_gpu=sb)


def test_fused_append_full_size_step(K):
    """One decode step of a full Qwen3-4B-shaped layer (batch 16, 1024 blocks of
    32 tokens, 8 KV heads of d 128) in the launch configuration of the bench."""
    w = C3
    B = w.block_size
    mb = w.n_blocks + 6
    x = to_dev(generate_layer(w, 0, max_blocks=mb), "cuda:0")
    k = w.ks[0]
    xb = dict(x, kv_pages=x["kv_pages"].clone())
    da, db = _decoder(w, mb, k), _decoder(w, mb, k)
    sa, aa = da.new_summaries()
    sb, ab = db.new_summaries()
    da.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], sa, aa)
    db.build_summaries(xb["kv_pages"], x["block_table"], x["seq_lens"], sb, ab)
    g = torch.Generator(device="cuda:0")
    g.manual_seed(3)
    shape = (w.batch, w.n_kvheads, w.head_dim)
    new_k = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
    new_v = torch.randn(shape, generator=g, device="cuda:0").to(torch.bfloat16)
    pos = x["seq_lens"].clone()
    nxt = pos + 1
    sc_a = torch.zeros((w.batch, mb), device="cuda:0")
    sc_b = torch.zeros((w.batch, mb), device="cuda:0")
    da.append(x["kv_pages"], x["block_table"], pos, sa, aa, new_k=new_k, new_v=new_v)
    da.select(x["q"], sa, nxt, scores_out=sc_a)
    db.append_select(xb["kv_pages"], x["block_table"], pos, x["q"], sb, ab, nxt, new_k=new_k,
                     new_v=new_v, scores_out=sc_b)
    torch.cuda.synchronize()
    assert _same(x["kv_pages"], xb["kv_pages"])
    assert _same(sa, sb) and _same(aa, ab)
    n = (int(nxt[0]) + B - 1) // B
    assert _same(sc_a[:, :n], sc_b[:, :n])
    assert torch.equal(da.n_sel, db.n_sel) and torch.equal(da.sel_idx, db.sel_idx)
    assert torch.equal(da.n_spans, db.n_spans) and torch.equal(da.dense_flag, db.dense_flag)


def test_fused_append_position_out_of_range(K):
    """A position past the table latches BOUNDS once and changes nothing, as the
    APPEND call does; the other sequences are served."""
    w = C0.scaled(batch=3, seq_len=100)
    mb = 8
    x = to_dev(generate_layer(w, 0, max_blocks=mb, seq_lens=[100, 90, 60]), "cuda:0")
    xb = dict(x, kv_pages=x["kv_pages"].clone())
    da, db = _decoder(w, mb, 3), _decoder(w, mb, 3)
    sa, aa = da.new_summaries()
    sb, ab = db.new_summaries()
    da.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], sa, aa)
    db.build_summaries(xb["kv_pages"], x["block_table"], x["seq_lens"], sb, ab)
    new_k = torch.ones((w.batch, w.n_kvheads, w.head_dim), dtype=torch.bfloat16, device="cuda:0")
    pos = torch.tensor([100, mb * w.block_size, 60], dtype=torch.int32, device="cuda:0")
    nxt = torch.tensor([101, 90, 61], dtype=torch.int32, device="cuda:0")
    da.append(x["kv_pages"], x["block_table"], pos, sa, aa, new_k=new_k, new_v=new_k)
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS
    da.select(x["q"], sa, nxt)
    db.append_select(xb["kv_pages"], x["block_table"], pos, x["q"], sb, ab, nxt, new_k=new_k,
                     new_v=new_k)
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS
    assert _same(x["kv_pages"], xb["kv_pages"]) and _same(sa, sb) and _same(aa, ab)
    assert torch.equal(da.sel_idx, db.sel_idx) and torch.equal(da.n_sel, db.n_sel)
