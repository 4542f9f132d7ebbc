"""The block-mean division of the summary kernels is IEEE division.

A block summary is the fp64 sum of the block's keys divided by the token
count and rounded once to bf16 ("SparPR KV cache recovery on a consumer GPU",
paragraph "Query-Aware key-block selection": the summary is the block's mean
key). The kernels divide with one correctly rounded reciprocal 1/c, the
product q = x * (1/c), its exact residual x - q*c and one correction step
(Markstein's division) instead of an fp64 division per channel. That is the
correctly rounded quotient, which the bit-exact summaries rely on; here it is
checked against IEEE fp64 division (numpy) bit for bit through
kvsel_selftest_divide on:
  * block sums as the summaries form them: the sequential fp64 sum from +0.0
    of 1 to 64 bf16 keys, drawn at scales from bf16's subnormals to its
    largest finite values, mixed within a block, with cancellation;
  * every count from 1 to 64 for each kind of sum;
  * signed zeros, infinities and NaN.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


def _bf16_values(rng, n, scale_exp):
    """n bf16 values (as float64) with magnitudes around 2^scale_exp."""
    mant = rng.integers(128, 256, n).astype(np.float64) / 128.0          # [1, 2) on the bf16 grid
    exp = scale_exp + rng.integers(-6, 7, n)
    x = np.ldexp(mant, exp) * np.where(rng.random(n) < 0.5, -1.0, 1.0)
    with np.errstate(over="ignore"):            # the largest scales reach bf16's infinities
        x = x.astype(np.float32)
    bits = x.view(np.uint32) & np.uint32(0xFFFF0000)                  # already on the grid; drop nothing
    return bits.view(np.float32).astype(np.float64)


def _block_sums(rng, blocks, counts, scale_exps):
    """The sequential fp64 sum from +0.0 of count[i] bf16 keys per block."""
    out = np.empty(blocks, np.float64)
    for i in range(blocks):
        vals = _bf16_values(rng, counts[i], scale_exps[i])
        acc = 0.0
        with np.errstate(over="ignore", invalid="ignore"):   # sums may reach inf, inf - inf = NaN
            for v in vals:
                acc = acc + v
        out[i] = acc
    return out


def _check(K, x, cnt):
    xd = torch.from_numpy(x).to("cuda:0")
    cd = torch.from_numpy(cnt.astype(np.int32)).to("cuda:0")
    out = torch.empty_like(xd)
    K.kvsel_selftest_divide(xd, cd, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = x / cnt.astype(np.float64)
    same = (got.view(np.uint64) == want.view(np.uint64)) | (np.isnan(got) & np.isnan(want))
    bad = np.flatnonzero(~same)
    assert bad.size == 0, [(x[i], int(cnt[i]), got[i], want[i]) for i in bad[:5]]


def test_division_of_block_sums_is_ieee(K):
    rng = np.random.default_rng(7)
    blocks = 20000
    counts = rng.integers(1, 65, blocks)
    # scales from bf16 subnormals (2^-133) to near its largest finite values (2^127)
    scale_exps = rng.choice(np.array([-133, -126, -100, -30, -8, 0, 3, 20, 60, 100, 120, 126]), blocks)
    sums = _block_sums(rng, blocks, counts, scale_exps)
    # every count 1..64 against every sum
    x = np.repeat(sums, 64)
    cnt = np.tile(np.arange(1, 65), blocks)
    _check(K, x, cnt)


def test_division_of_wide_sums_and_special_values(K):
    rng = np.random.default_rng(11)
    n = 1 << 22
    # sums whose keys span a wide range of exponents (the kernels then add in
    # fp64), and dense random fp64 values of the same magnitudes
    x = np.ldexp(rng.random(n) + 1.0, rng.integers(-140, 134, n)) * np.where(rng.random(n) < 0.5, -1.0, 1.0)
    x = np.concatenate([x, np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 2.0 ** -133, -(2.0 ** 134),
                                     3.3895313892515355e38 * 64])])
    cnt = rng.integers(1, 65, x.size)
    _check(K, x, cnt)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan])
    for c in range(1, 65):
        _check(K, special, np.full(special.size, c))
