"""GPU: the block cache of the host tier (kvsel_cache_reset / kvsel_cache_fetch)
against the oracle's BlockCache state machine, bit for bit on the cache state
and the copied pages over many steps, and end to end on a MiniCPM-shaped
offload problem: select, fetch through the cache, attend over the pool,
against the uncached host path (bit for bit) and the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle as o
from tests._parity import attn_errors, selection_verdict
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


def _selections(g, N, k, locality):
    sel = np.sort(g.choice(N, size=k, replace=False))
    while True:
        keep = sel[g.random(len(sel)) < locality]
        rest = np.setdiff1d(np.arange(N), keep)
        kk = int(g.integers(max(1, len(keep)), k + 1))
        sel = np.sort(np.concatenate([keep[:kk], g.choice(rest, size=kk - min(kk, len(keep)), replace=False)]))
        yield sel


@pytest.mark.parametrize("slots,locality", [(8, 0.6), (11, 0.8), (24, 0.3)])
def test_cache_state_and_pages_match_the_oracle_over_many_steps(K, slots, locality):
    from query_aware_sparse_block_gb300.runtime import HostBlockCache, SparseDecoder
    w = C0.scaled(batch=3, seq_len=64 * 16)
    N, k = 64, 8
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, N, k_max=k,
                        device="cuda:0")
    page = (w.n_kvheads, 2, w.head_dim // 64, w.block_size, 64)
    g = torch.Generator().manual_seed(slots)
    host = torch.randn((w.batch, N) + page, generator=g).to(torch.bfloat16).pin_memory()
    cache = HostBlockCache(dec, slots, page)
    seq_lens = torch.full((w.batch,), N * w.block_size, dtype=torch.int32, device="cuda:0")
    ref = [o.BlockCache(slots) for _ in range(w.batch)]
    rng = np.random.default_rng(slots)
    gens = [_selections(rng, N, k, locality) for _ in range(w.batch)]
    fetched_total = 0
    for step in range(40):
        sels = [next(gens[b]) for b in range(w.batch)]
        if step % 3 == 0:
            sels[0] = np.union1d(sels[0][: k - 1], [N - 1])      # the open block selected
        sel = torch.zeros((w.batch, k), dtype=torch.int32)
        for b in range(w.batch):
            sel[b, : len(sels[b])] = torch.from_numpy(sels[b].astype(np.int32))
        n_sel = torch.tensor([len(s) for s in sels], dtype=torch.int32)
        # an append rewrites the open block of sequence 0 in the host tier
        host[0, N - 1].copy_(torch.randn(page, generator=g).to(torch.bfloat16))
        cache.fetch(host, N, seq_lens, sel.to("cuda:0"), n_sel.to("cuda:0"))
        torch.cuda.synchronize()
        nf = cache.n_fetched.cpu().tolist()
        page_of = cache.page_of.cpu()
        for b in range(w.batch):
            jobs, _ = ref[b].step(sels[b], step, N - 1)
            assert nf[b] == len(jobs), (step, b)
            fetched_total += nf[b]
            assert cache.block_in[b].cpu().tolist() == ref[b].block_in, (step, b)
            assert cache.last_use[b].cpu().tolist() == ref[b].last_use, (step, b)
            want = torch.full((N,), -1, dtype=torch.int32)
            for blk, s in ref[b].slot_of.items():
                want[blk] = b * slots + s
            assert torch.equal(page_of[b], want), (step, b)
            for blk, s in ref[b].slot_of.items():
                if b == 0 and blk == N - 1 and blk not in sels[b]:
                    continue                    # stale until selected again (then re-fetched)
                assert torch.equal(cache.pool[b * slots + s].cpu().view(torch.int16),
                                   host[b, blk].view(torch.int16)), (step, b, blk)
    assert 0 < fetched_total < 40 * w.batch * k         # some reuse, some traffic


def test_cache_rejects_a_selection_that_is_not_ascending(K):
    from query_aware_sparse_block_gb300.runtime import HostBlockCache, SparseDecoder
    w = C0.scaled(batch=1, seq_len=320)
    dec = SparseDecoder(1, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, 20, k_max=4,
                        device="cuda:0")
    page = (w.n_kvheads, 2, w.head_dim // 64, w.block_size, 64)
    host = torch.zeros((1, 20) + page, dtype=torch.bfloat16).pin_memory()
    cache = HostBlockCache(dec, 4, page)
    sel = torch.tensor([[3, 2, 7, 9]], dtype=torch.int32, device="cuda:0")
    cache.fetch(host, 20, torch.tensor([320], dtype=torch.int32, device="cuda:0"), sel,
                torch.tensor([4], dtype=torch.int32, device="cuda:0"))
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS
    # the entries that break the order are not served; the others are cached
    assert sorted(b for b in cache.block_in[0].cpu().tolist() if b >= 0) == [3, 7, 9]


def test_offload_through_the_cache_equals_the_uncached_path_and_the_oracle(K):
    """MiniCPM4.1-8B-shaped host tier (32 q / 2 KV heads, d 128, 131072 tokens
    in blocks of 64) for 4 sequences; queries drift from step to step
    (q_s = 0.95 q_(s-1) + 0.31 e_s), so consecutive selections overlap."""
    from query_aware_sparse_block_gb300.runtime import HostBlockCache, SparseDecoder
    w = C4.scaled(batch=4)
    N = w.n_blocks
    k = w.k_for(w.keep_floor)
    x = generate_layer(w, 0, device="cuda:0", perm=False)
    page = tuple(x["kv_pages"].shape[1:])
    host = torch.empty((w.batch, N) + page, dtype=torch.bfloat16, pin_memory=True)
    host_tier_layout(x["kv_pages"], x["block_table"], N, out=host)
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, N, k_max=k,
                        device="cuda:0")
    ref_dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, N, k_max=k,
                            device="cuda:0")
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    del x["kv_pages"]
    torch.cuda.empty_cache()
    dec.k_per_seq.fill_(k)
    cache = HostBlockCache(dec, 2 * k, page)
    staging = torch.empty((w.batch, k) + page, dtype=torch.bfloat16, device="cuda:0")
    kv_host = K.kv_host(host, N, staging, k)
    g = torch.Generator(device="cuda:0").manual_seed(77)
    q = x["q"].float()
    rho = 0.95
    oref = [o.BlockCache(2 * k) for _ in range(w.batch)]
    fetched = []
    for step in range(4):
        if step:
            q = rho * q + math.sqrt(1 - rho * rho) * torch.randn(q.shape, generator=g, device="cuda:0")
        qb = q.to(torch.bfloat16)
        dec.select(qb, summ, x["seq_lens"])
        cache.fetch(host, N, x["seq_lens"], dec.sel_idx, dec.n_sel)
        dec.attend(qb, cache.kv, x["seq_lens"], use_dense_flag=False)
        # the uncached path on the same selection
        for name in ("sel_idx", "n_sel", "span_start", "span_len", "n_spans"):
            getattr(ref_dec, name).copy_(getattr(dec, name))
        ref_dec.attend(qb, kv_host, x["seq_lens"], use_dense_flag=False)
        torch.cuda.synchronize()
        assert torch.equal(dec.out, ref_dec.out) and torch.equal(dec.lse, ref_dec.lse), step
        nf = cache.n_fetched.cpu().tolist()
        fetched.append(sum(nf))
        for b in range(w.batch):
            gsel = dec.sel_idx[b, : int(dec.n_sel[b])].cpu().numpy()
            jobs, _ = oref[b].step(gsel, step, N - 1)
            assert nf[b] == len(jobs)
        if step in (0, 3):
            b = step % w.batch
            qbits = bits(qb[b])
            kb = bits(natural_blocks(host[b, :, :, 0]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
            vb = bits(natural_blocks(host[b, :, :, 1]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
            sb, _, _ = o.block_summaries(kb, w.seq_len, w.block_size)
            gsel = dec.sel_idx[b, : int(dec.n_sel[b])].cpu().numpy()
            selection_verdict(o.block_scores(qbits, sb), k, gsel)
            ref, _ = o.attend(qbits, kb, vb, o.tokens_of_blocks(gsel, w.seq_len, w.block_size), dec.scale)
            emax, emean = attn_errors(dec.out[b].cpu().numpy(), ref)
            assert emax <= 1e-2 and emean <= 1e-3, (step, b, emax, emean)
    assert fetched[0] == w.batch * k
    assert all(f < w.batch * k for f in fetched[1:]), fetched    # drifting queries reuse blocks
