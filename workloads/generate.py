"""Seeded synthetic inputs shared by the tests, the bench and the oracle.

This module draws random numbers and lays tensors out; it holds none of the
method's arithmetic (no summaries, scores, selection or attention).

Recipe (per layer): a ``torch.Generator`` seeded with ``Workload.seed(layer)``
draws q, then K, then V, each ~N(0, 1) in fp32 and rounded to bf16. Then:
  * needles: for every listed block n and every token of it, the key of KV
    head j is bf16(4 * q[first query head of j's group]) (a power-of-two scale,
    so it is exact);
  * outlier channels: K[..., j, c] *= scale for c < outlier_channels;
  * drift: K[t, j, c] += amp * sin(2*pi*t/period + 2*pi*(j*d + c)/(H_kv*d)),
    added in fp32 before the bf16 rounding.

Device layout (paged cache): one KV page array [n_pages][H_kv][2][d/64][B][64]
bf16 -- for each (page, KV head) the K tile, then the V tile; each tile stores
its B x d values as d/64 column halves of B rows x 64 channels, and within
every 128-byte row the 16-byte chunk c of token row t sits at chunk position
c ^ (t % 8). ``to_tiled`` / ``from_tiled`` convert between a tile and the
natural [..., B, d] order. The block table [batch][max_blocks] int32 maps a
sequence's logical block to its page. ``perm=True`` scatters logical blocks
over pages in a seeded random order so that every path goes through the
table.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .configs import Workload


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _chunk_swizzle(y: torch.Tensor) -> torch.Tensor:
    """[..., B, 8 chunks, 8] -> same shape with chunk c of row t moved to c ^ (t % 8).

    XOR is its own inverse, so the same routine un-swizzles.
    """
    B = y.shape[-3]
    out = torch.empty_like(y)
    for r in range(8):
        perm = torch.tensor([c ^ r for c in range(8)], device=y.device)
        out[..., r::8, :, :] = y[..., r::8, :, :].index_select(-2, perm)
    return out


def to_tiled(x: torch.Tensor) -> torch.Tensor:
    """Natural [..., B, d] tiles -> the cache layout [..., d/64, B, 64]."""
    *lead, B, d = x.shape
    h2 = d // 64
    y = x.reshape(*lead, B, h2, 8, 8).movedim(-3, -4)        # [..., h2, B, 8, 8]
    return _chunk_swizzle(y).reshape(*lead, h2, B, 64)


def from_tiled(y: torch.Tensor) -> torch.Tensor:
    """Cache layout [..., d/64, B, 64] -> natural [..., B, d]."""
    *lead, h2, B, _ = y.shape
    x = _chunk_swizzle(y.reshape(*lead, h2, B, 8, 8))        # [..., h2, B, 8, 8]
    return x.movedim(-4, -3).reshape(*lead, B, h2 * 64)


def generate_layer(w: Workload, layer: int = 0, device="cpu", max_blocks: int | None = None,
                   perm: bool = True, seq_lens=None, seed: int | None = None) -> dict:
    """Inputs of one layer of one decode step.

    Returns dict with q [b][H_q][d] bf16, kv_pages [n_pages][H_kv][2][d/64][B][64]
    bf16, block_table [b][max_blocks] int32 and seq_lens [b] int32 (all on
    ``device``). ``max_blocks`` may exceed the blocks in use (room to append).
    """
    b, Hq, Hkv, d, B = w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size
    N = w.n_blocks
    MB = max(N, max_blocks or 0)
    g = _gen(w.seed(layer) if seed is None else seed, device)
    q32 = _randn_bf16((b, Hq, d), g, device)
    q = q32.to(torch.bfloat16)
    # K and V are drawn in the logical blocked layout [b][MB][H_kv][B][d].
    k32 = _randn_bf16((b, MB, Hkv, B, d), g, device)
    if w.outlier_channels:
        k32[..., : w.outlier_channels] *= w.outlier_scale
    if w.drift_amp:
        t = torch.arange(MB * B, device=device, dtype=torch.float32).view(MB, 1, B, 1)
        jc = (torch.arange(Hkv, device=device, dtype=torch.float32).view(1, Hkv, 1, 1) * d
              + torch.arange(d, device=device, dtype=torch.float32).view(1, 1, 1, d))
        phase = 2 * math.pi * t / w.drift_period + 2 * math.pi * jc / (Hkv * d)
        k32 += w.drift_amp * torch.sin(phase).unsqueeze(0)
        del t, jc, phase
    kb = k32.to(torch.bfloat16)
    del k32
    if w.needles:
        G = Hq // Hkv
        needle_key = (4.0 * q32[:, ::G, :]).to(torch.bfloat16)  # [b][H_kv][d]
        for n in w.needles:
            kb[:, n] = needle_key[:, :, None, :].expand(b, Hkv, B, d)
    vb = _randn_bf16((b, MB, Hkv, B, d), g, device).to(torch.bfloat16)
    n_pages = b * MB
    if perm:
        gp = _gen((w.seed(layer) if seed is None else seed) + 7919, "cpu")
        page_of = torch.randperm(n_pages, generator=gp).to(torch.int32)
    else:
        page_of = torch.arange(n_pages, dtype=torch.int32)
    block_table = page_of.view(b, MB).to(device)
    kv_pages = torch.empty((n_pages, Hkv, 2, d // 64, B, 64), dtype=torch.bfloat16, device=device)
    idx = page_of.to(device=device, dtype=torch.long)
    kv_pages[idx, :, 0] = to_tiled(kb.view(n_pages, Hkv, B, d))
    del kb
    kv_pages[idx, :, 1] = to_tiled(vb.view(n_pages, Hkv, B, d))
    del vb
    if seq_lens is None:
        seq_lens = torch.full((b,), w.seq_len, dtype=torch.int32)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).to(device)
    return dict(q=q, kv_pages=kv_pages, block_table=block_table.contiguous(),
                seq_lens=seq_lens, max_blocks=MB)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (a reinterpretation, no rounding)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def logical_kv(kv_pages: torch.Tensor, block_table: torch.Tensor, b: int, T: int,
               which: int) -> torch.Tensor:
    """One sequence's keys (which=0) or values (which=1) in token order [T][H_kv][d]."""
    B = kv_pages.shape[4]
    N = (T + B - 1) // B
    p = block_table[b, :N].long().to(kv_pages.device)
    blk = from_tiled(kv_pages[p][:, :, which])      # [N][H_kv][B][d]
    return blk.permute(0, 2, 1, 3).reshape(N * B, blk.shape[1], blk.shape[3])[:T]


def natural_blocks(tiles: torch.Tensor) -> torch.Tensor:
    """[..., H_kv, d/64, B, 64] cache tiles -> token-major [..., B, H_kv, d]."""
    x = from_tiled(tiles)                           # [..., H_kv, B, d]
    return x.transpose(-3, -2)


def host_tier_layout(kv_pages: torch.Tensor, block_table: torch.Tensor, n_blocks: int,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """Offload-tier layout [b][N][one page]: block n of sequence s is page block_table[s][n]."""
    b = block_table.shape[0]
    if out is None:
        out = torch.empty((b, n_blocks) + tuple(kv_pages.shape[1:]), dtype=torch.bfloat16)
    for s in range(b):
        p = block_table[s, :n_blocks].long().to(kv_pages.device)
        out[s].copy_(kv_pages[p])
    return out
