"""GPU: the FULL summary build on every bf16 bit pattern. 128 blocks of 16
identical tokens (8 KV heads x 64 channels) carry all 65536 patterns, one per
column, so each summary is the mean of 16 copies of one value and each
open-block sum is 16 times it; both are compared bit for bit with the fp64
oracle (NaN patterns only as NaN). This pins the widening of bf16 to fp64 in
the summary arithmetic for normal, subnormal, zero and infinite values."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as o
from workloads import C0
from workloads.generate import bits, to_tiled

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


def _is_nan(b):
    return ((b >> 7) & 0xFF == 0xFF) & ((b & 0x7F) != 0)


@pytest.mark.parametrize("batch", [1, 3])
def test_every_bf16_pattern_through_the_full_build(K, batch):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    w = C0
    H, d, B = w.n_kvheads, w.head_dim, w.block_size
    N = 65536 // (H * d)                                    # 128 blocks
    pat = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(N, H, d)
    keys = np.broadcast_to(pat[:, :, None, :], (N, H, B, d))            # [N][H][B][d]
    kb = torch.from_numpy(np.ascontiguousarray(keys).view(np.int16)).view(torch.bfloat16)
    pages = torch.zeros((batch * N, H, 2, d // 64, B, 64), dtype=torch.bfloat16)
    for s in range(batch):
        pages[s * N:(s + 1) * N, :, 0] = to_tiled(kb)
    dev = "cuda:0"
    pages = pages.to(dev)
    # sequence s uses its own pages; the last sequence ends mid-block
    table = torch.arange(batch * N, dtype=torch.int32).view(batch, N).to(dev)
    lens = [N * B] * batch
    lens[-1] = N * B - 5
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=dev)
    dec = SparseDecoder(batch, w.n_qheads, H, d, B, N, k_max=1, device=dev)
    summ, acc = dec.new_summaries()
    dec.build_summaries(pages, table, seq_lens, summ, acc)
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == 0
    for s in range(batch):
        T = lens[s]
        kseq = np.ascontiguousarray(np.broadcast_to(pat[:, None, :, :], (N, B, H, d))).reshape(N * B, H, d)[:T]
        want, _, last = o.block_summaries(kseq, T, B)
        got = bits(summ[s])
        nan_w, nan_g = _is_nan(want), _is_nan(got)
        assert np.array_equal(nan_w, nan_g), f"NaN positions differ (seq {s})"
        assert np.array_equal(np.where(nan_w, 0, want), np.where(nan_g, 0, got)), f"summaries differ (seq {s})"
        a = acc[s].cpu().numpy()
        assert np.array_equal(np.isnan(a), np.isnan(last))
        fin = ~np.isnan(last)
        assert np.array_equal(a[fin], last[fin]), f"open-block sums differ (seq {s})"
