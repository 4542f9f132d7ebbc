"""GPU: a decode step driven from plain C (tests/gpu_c_consumer.c: cudaMalloc'd
buffers, the C ABI, no PyTorch in the process) on ragged sequences spanning
several tiles, checked against the fp64 oracle: selection by the tie rule,
attention within the stated tolerance."""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle as o
from tests._parity import ATOL_MAX, ATOL_MEAN, attn_errors, seq_inputs, selection_verdict
from workloads import C3
from workloads.generate import bits, generate_layer

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from query_aware_sparse_block_gb300.build import LIB, build_library
    build_library()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    path = str(tmp_path_factory.mktemp("c") / "gpu_c_consumer")
    libdir = os.path.dirname(LIB)
    subprocess.run([nvcc, "-x", "c", "-O2", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "gpu_c_consumer.c"), "-L", libdir, "-lkvsel",
                    "-Xlinker", "-rpath," + libdir, "-lm", "-o", path], check=True)
    return path


def test_c_program_decode_step_matches_the_oracle(exe, tmp_path):
    w = C3.scaled(batch=3, seq_len=2000, drift_amp=0.0, layers=1)
    lens = [2000, 777, 1]
    k = 9
    x = generate_layer(w, 0, seq_lens=lens)          # CPU tensors, scattered pages
    n_pages = x["kv_pages"].shape[0]
    hdr = np.array([w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, x["max_blocks"], k,
                    n_pages], dtype=np.int32)
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        f.write(hdr.tobytes())
        f.write(bits(x["q"]).tobytes())
        f.write(bits(x["kv_pages"]).tobytes())
        f.write(x["block_table"].numpy().astype(np.int32).tobytes())
        f.write(x["seq_lens"].numpy().astype(np.int32).tobytes())
    r = subprocess.run([exe, str(fin), str(fout)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = np.fromfile(fout, dtype=np.uint8)
    B, H, d = w.batch, w.n_qheads, w.head_dim
    o0 = B * k * 4
    o1 = o0 + B * 4
    o2 = o1 + B * H * d * 4
    sel = raw[:o0].view(np.int32).reshape(B, k)
    n_sel = raw[o0:o1].view(np.int32)
    out = raw[o1:o2].view(np.float32).reshape(B, H, d)
    lse = raw[o2:].view(np.float32).reshape(B, H)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    for b in range(B):
        T = lens[b]
        qb, kb, vb = seq_inputs(x, b, T)
        sb = o.block_summaries(kb, T, w.block_size)[0]
        scores = o.block_scores(qb, sb)
        gsel = sel[b, : n_sel[b]].astype(np.int64)
        selection_verdict(scores, k, gsel)
        ref, ref_lse = o.attend(qb, kb, vb, o.tokens_of_blocks(gsel, T, w.block_size), scale)
        emax, emean = attn_errors(out[b].astype(np.float64), ref)
        assert emax <= ATOL_MAX and emean <= ATOL_MEAN, (b, emax, emean)
        assert np.abs(lse[b] - ref_lse).max() <= 1e-3 * max(1.0, np.abs(ref_lse).max())
