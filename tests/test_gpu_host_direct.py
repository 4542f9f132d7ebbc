"""GPU: kvsel_sparse_decode reading the host tier directly (KVSEL_KV_HOST_DIRECT,
16-byte asynchronous copies from pinned host memory into the attention
kernel's shared memory, no staging) against the same kernel reading the
device pages (bit for bit: the same tiles land in the same order), against
the staged host path on a MiniCPM-shaped offload problem (bit for bit) and
against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as o
from tests._parity import attn_errors, check_sequence, selection_verdict, to_dev
from workloads import C0, C2, C3, C4
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


def _decoder(w, mb, k_max=None):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    return SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, mb, k_max=k_max,
                         device="cuda:0")


CASES = [
    # name, workload, seq_lens, k, gamma
    ("mha_d64_B16_ragged", C0.scaled(batch=4, seq_len=1000), [1000, 37, 0, 513], 7, 2.0),
    ("gqa4_d128_B32_dense_one", C3.scaled(batch=3, seq_len=2000, drift_amp=0.0, layers=1), [2000, 100, 1999], 4, 0.9),
    ("gqa16_d128_B64", C2.scaled(batch=2, seq_len=9000, layers=1), [9000, 4097], 5, 2.0),
]


@pytest.mark.parametrize("name,w,lens,k,gamma", CASES, ids=[c[0] for c in CASES])
def test_host_direct_equals_device_pages_bit_for_bit(K, name, w, lens, k, gamma):
    x = to_dev(generate_layer(w, 0, seq_lens=lens), "cuda:0")
    mb = x["max_blocks"]
    dec = _decoder(w, mb)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.fill_(k)
    dec.select(x["q"], summ, x["seq_lens"], gamma=gamma)
    host = torch.empty((w.batch, mb) + tuple(x["kv_pages"].shape[1:]), dtype=torch.bfloat16,
                       pin_memory=True)
    host_tier_layout(x["kv_pages"], x["block_table"], mb, out=host)
    dec.attend(x["q"], K.kv_paged(x["kv_pages"], x["block_table"]), x["seq_lens"])
    out_p, lse_p = dec.out.clone(), dec.lse.clone()
    dec.out.zero_()
    dec.attend(x["q"], K.kv_host_direct(host, mb), x["seq_lens"])
    torch.cuda.synchronize()
    assert torch.equal(dec.out, out_p) and torch.equal(dec.lse, lse_p)
    if gamma < 1.0:
        assert bool(dec.dense_flag[1])            # 4 of 4 blocks of the short sequence
    for b in range(w.batch):
        check_sequence(dec, x, b, lens[b], w.block_size, k, dec.scale, gamma=gamma)


def test_host_direct_block_past_the_host_tier_is_latched(K):
    w = C0.scaled(batch=1, seq_len=320)
    x = to_dev(generate_layer(w, 0), "cuda:0")
    dec = _decoder(w, x["max_blocks"], k_max=4)
    dec.n_sel.fill_(3)
    dec.sel_idx[0, :3] = torch.tensor([1, 5, 19], dtype=torch.int32)
    host = torch.zeros((1, 12) + tuple(x["kv_pages"].shape[1:]), dtype=torch.bfloat16, pin_memory=True)
    dec.attend(x["q"], K.kv_host_direct(host, 12), x["seq_lens"], use_dense_flag=False)
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == K.KVSEL_ERR_BOUNDS


def test_minicpm_offload_host_direct_equals_staged_and_oracle(K):
    """MiniCPM4.1-8B-shaped host tier (4 sequences of 131072 tokens, 32 q / 2
    KV heads, d 128, blocks of 64, keep floor 5 %)."""
    w = C4.scaled(batch=4)
    N = w.n_blocks
    k = w.k_for(w.keep_floor)
    x = generate_layer(w, 0, device="cuda:0", perm=False)
    page = tuple(x["kv_pages"].shape[1:])
    host = torch.empty((w.batch, N) + page, dtype=torch.bfloat16, pin_memory=True)
    host_tier_layout(x["kv_pages"], x["block_table"], N, out=host)
    dec = _decoder(w, N, k_max=k)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    del x["kv_pages"]
    torch.cuda.empty_cache()
    dec.k_per_seq.fill_(k)
    dec.select(x["q"], summ, x["seq_lens"], gamma=w.gamma)
    staging = torch.empty((w.batch, k) + page, dtype=torch.bfloat16, device="cuda:0")
    dec.attend(x["q"], K.kv_host(host, N, staging, k), x["seq_lens"])
    out_s, lse_s = dec.out.clone(), dec.lse.clone()
    dec.out.zero_()
    dec.attend(x["q"], K.kv_host_direct(host, N), x["seq_lens"])
    torch.cuda.synchronize()
    assert torch.equal(dec.out, out_s) and torch.equal(dec.lse, lse_s)
    b = 2
    qb = bits(x["q"][b])
    kb = bits(natural_blocks(host[b, :, :, 0]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
    vb = bits(natural_blocks(host[b, :, :, 1]).reshape(N * w.block_size, w.n_kvheads, w.head_dim))
    sb, _, _ = o.block_summaries(kb, w.seq_len, w.block_size)
    gsel = dec.sel_idx[b, : int(dec.n_sel[b])].cpu().numpy()
    selection_verdict(o.block_scores(qb, sb), k, gsel)
    ref, _ = o.attend(qb, kb, vb, o.tokens_of_blocks(gsel, w.seq_len, w.block_size), dec.scale)
    emax, emean = attn_errors(dec.out[b].cpu().numpy(), ref)
    assert emax <= 1e-2 and emean <= 1e-3, (emax, emean)
