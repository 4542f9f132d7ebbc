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


def _column_mix(rng, n_blocks, H, B, d):
    """Keys [n_blocks][H][B][d] whose block columns exercise every path of
    the summary sum: exponents within a narrow range (the exact integer
    sum), a range wider than 2^39 (the sequential fp64 sum, which rounds),
    exact cancellation, and an infinity or a NaN among finite values."""
    x = rng.standard_normal((n_blocks, H, B, d))
    kind = rng.integers(0, 5, (n_blocks, H, 1, d))
    narrow = np.ldexp(x, rng.integers(-15, 16, x.shape))
    wide = np.ldexp(x, rng.integers(-90, 91, x.shape))
    cancel = np.concatenate([x[:, :, : B // 2], -x[:, :, : B // 2]], axis=2)
    special = x.copy()
    special[:, :, B // 3] = np.where(rng.random((n_blocks, H, d)) < 0.5, np.inf, np.nan)
    special[:, :, B // 5] = np.where(rng.random((n_blocks, H, d)) < 0.2, -np.inf, special[:, :, B // 5])
    out = np.select([kind == 0, kind == 1, kind == 2, kind == 3], [x, narrow, wide, cancel], special)
    return torch.from_numpy(out.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.filterwarnings("ignore:invalid value encountered:RuntimeWarning")   # inf + -inf columns
@pytest.mark.parametrize("H,d,B", [(8, 64, 16), (2, 128, 64)])
def test_summary_sum_paths_match_the_oracle(K, H, d, B):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    rng = np.random.default_rng(H * 1000 + B)
    N, batch = 48, 2
    kb = _column_mix(rng, batch * N, H, B, d)                  # [pages][H][B][d]
    dev = "cuda:0"
    pages = torch.zeros((batch * N, H, 2, d // 64, B, 64), dtype=torch.bfloat16)
    pages[:, :, 0] = to_tiled(kb)
    perm = torch.from_numpy(rng.permutation(batch * N).astype(np.int32))
    pages = pages[perm.argsort()]                             # page perm[i] holds logical block i
    table = perm.view(batch, N).to(dev)
    lens = [N * B, N * B - B // 2 - 1]                         # the second ends mid-block
    dec = SparseDecoder(batch, 4 * H, H, d, B, N, k_max=1, device=dev)
    summ, acc = dec.new_summaries()
    dec.build_summaries(pages.to(dev), table, torch.tensor(lens, dtype=torch.int32, device=dev), summ, acc)
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == 0
    for s in range(batch):
        T = lens[s]
        kseq = bits(kb[s * N:(s + 1) * N].permute(0, 2, 1, 3).reshape(N * B, H, d))[:T]
        want, _, last = o.block_summaries(kseq, T, B)
        got = bits(summ[s])
        nan_w, nan_g = _is_nan(want), _is_nan(got)
        assert np.array_equal(nan_w, nan_g), f"NaN positions differ (seq {s})"
        assert np.array_equal(np.where(nan_w, 0, want), np.where(nan_g, 0, got)), f"summaries differ (seq {s})"
        a = acc[s].cpu().numpy()
        assert np.array_equal(np.isnan(a), np.isnan(last))
        fin = ~np.isnan(last)
        assert np.array_equal(a[fin], last[fin]), f"open-block sums differ (seq {s})"
