"""Synthetic decode-step workloads (shapes only; no method arithmetic here).

The shapes follow the models the pages evaluate on:
  C0  tiny MHA smoke case.
  C1  OPT-6.7B-shaped MHA ("SparPR KV cache recovery on a consumer GPU",
      section "Measured numbers on one laptop": facebook/opt-6.7b, batch 4,
      a needle planted at two depths, keep ratios 50 % and 10 %).
  C2  MiniCPM4.1-8B-shaped GQA ("KV cache offloading", section "Why the cache
      leaves the GPU": 32 layers, 32 heads, 2 KV heads, head dim 128, 131 072
      tokens) at the 3.13 % resident share of the VerKV article.
  C3  Qwen3-4B-shaped GQA batch decode (VerKV article, section "Perspective":
      Qwen3-4B at 32K context, 12.5 % resident share).
  C4  offload tier: the MiniCPM4.1-8B shape at batch 64 ("KV cache
      offloading", sections "Why the cache leaves the GPU" and "SparDA").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    batch: int
    n_qheads: int
    n_kvheads: int
    head_dim: int
    seq_len: int
    block_size: int
    layers: int
    keep: tuple = ()            # keep ratios; k = clamp(floor(r*N + 1/2), 1, N)
    topk: int | None = None     # explicit k (overrides keep)
    needles: tuple = ()         # block indices whose keys are set to 4*q
    outlier_channels: int = 0   # first channels of each KV head scaled ...
    outlier_scale: float = 1.0  # ... by this factor
    drift_amp: float = 0.0      # K += amp * sin(2*pi*t/period + 2*pi*(j*d+c)/(H_kv*d))
    drift_period: int = 0
    offload: bool = False
    keep_floor: float = 0.0
    gamma: float = 1.0
    hidden: int = 0
    description: str = ""

    @property
    def n_blocks(self) -> int:
        return (self.seq_len + self.block_size - 1) // self.block_size

    @property
    def group(self) -> int:
        return self.n_qheads // self.n_kvheads

    def k_for(self, keep: float) -> int:
        N = self.n_blocks
        return max(1, min(N, int(math.floor(keep * N + 0.5))))

    @property
    def ks(self) -> tuple:
        if self.topk is not None:
            return (self.topk,)
        return tuple(self.k_for(r) for r in self.keep)

    def seed(self, layer: int = 0) -> int:
        return 0 if self.index == 0 else 1000 * self.index + layer

    def scaled(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


C0 = Workload("tiny_mha_b1_h8_d64_T1024_B16_k16", 0, 1, 8, 8, 64, 1024, 16, 1, topk=16,
              description="Tiny MHA decode step: batch 1, 8 heads, head_dim 64, 1024 tokens "
                          "in 64 blocks of 16, Top-k 16, one layer")
C1 = Workload("opt6.7b_mha_b4_h32_d128_T4096_B16", 1, 4, 32, 32, 128, 4096, 16, 32,
              keep=(0.5, 0.1), needles=(64, 192),
              description="OPT-6.7B-shaped MHA: batch 4, 32 heads, head_dim 128, 32 layers, "
                          "4096 tokens, block 16 (256 blocks), keep 50 % and 10 %, needle "
                          "blocks 64 and 192 with keys 4*q")
C2 = Workload("minicpm4.1-8b_gqa_b1_q32kv2_d128_T131072_B64", 2, 1, 32, 2, 128, 131072, 64, 1,
              keep=(0.0313,), outlier_channels=8, outlier_scale=10.0,
              description="MiniCPM4.1-8B-shaped GQA: batch 1, 32 q / 2 KV heads, head_dim 128, "
                          "131072 tokens, block 64 (2048 blocks), keep 3.13 % (64 blocks), "
                          "key channels 0-7 of each KV head scaled x10")
C3 = Workload("qwen3-4b_gqa_b16_q32kv8_d128_T32768_B32_keep12.5", 3, 16, 32, 8, 128, 32768, 32, 36,
              keep=(0.125,), drift_amp=1.0, drift_period=8192,
              description="Qwen3-4B-shaped GQA batch decode: batch 16, 32 q / 8 KV heads, "
                          "head_dim 128, 36 layers, 32768 tokens, block 32 (1024 blocks), "
                          "keep 12.5 % (128 blocks), K ~ N(0,1) + slow positional drift")
C4 = Workload("offload_minicpm_b64_q32kv2_d128_T131072_B64", 4, 64, 32, 2, 128, 131072, 64, 1,
              keep=(0.05, 0.125), offload=True, keep_floor=0.05, gamma=0.8, hidden=4096,
              description="Offload tier: batch 64, 32 q / 2 KV heads, head_dim 128, 131072 "
                          "tokens, block 64; K/V in pinned host memory, summaries on the GPU; "
                          "keep ratio from the copy/recompute model, floor 5 %, gamma 0.8")

ALL = (C0, C1, C2, C3, C4)
