"""GPU: failure detection without a fault. A bounded device wait that runs out
(a barrier phase nothing completes) must end with KVSEL_ERR_TIMEOUT in the
error word, read by kvsel_get_error on the host, and leave the context usable:
a decode step right after it matches the fp64 oracle."""
from __future__ import annotations

import time

import pytest
import torch

from tests._parity import check_sequence, to_dev
from workloads import C0
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


def test_a_wait_that_runs_out_reports_timeout_and_the_context_stays_usable(K):
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    assert K.kvsel_get_error() == 0
    t0 = time.perf_counter()
    K.kvsel_selftest_wait_timeout()
    assert K.kvsel_get_error() == K.KVSEL_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 1.9          # the wait limit is 2 s
    assert K.kvsel_get_error() == 0                 # read-and-clear
    w = C0
    x = to_dev(generate_layer(w, 0), "cuda:0")
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, x["max_blocks"],
                        device="cuda:0")
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    dec.k_per_seq.fill_(w.topk)
    dec.select(x["q"], summ, x["seq_lens"])
    dec.attend(x["q"], K.kv_paged(x["kv_pages"], x["block_table"]), x["seq_lens"])
    torch.cuda.synchronize()
    assert K.kvsel_get_error() == 0
    check_sequence(dec, x, 0, w.seq_len, w.block_size, w.topk, dec.scale, summaries_gpu=summ)
