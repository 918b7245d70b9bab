"""Seeded synthetic workloads for the attention forward pass.

This module holds only the input recipes (shapes, mask arguments, seeds, value
distributions) and the random number generation.  It contains none of the
attention arithmetic; both the CUDA path's tests/bench and the fp64 oracle take
their inputs from here, which is the one thing they share.

Recipe (every workload): Q, K, V drawn iid N(0, 1) in float32 from one seeded
CPU ``torch.Generator`` in the order Q, K, V (then any extra draws), then cast
once to the workload dtype; the same cast bits go to the GPU and, widened, to
the oracle.  scale = 1/sqrt(d_k) ("Trasformer 浅析", section 缩放因子的必要性).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch

MASK_FULL, MASK_CAUSAL, MASK_SLIDING, MASK_CAUSAL_SLIDING, MASK_LOCAL_GLOBAL = range(5)
MASK_NAMES = {MASK_FULL: "full", MASK_CAUSAL: "causal", MASK_SLIDING: "sliding",
              MASK_CAUSAL_SLIDING: "causal_sliding", MASK_LOCAL_GLOBAL: "local_global"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    d: int
    dtype: str          # "bf16" or "f32"
    kind: int
    window: int = 0
    globals_idx: Tuple[int, ...] = ()
    seed: int = 0
    q_upper_heads_scale: float = 1.0   # multiply Q heads [Hq/2, Hq) by this
    k_position_offset_std: float = 0.0  # add c_j ~ N(0, std) to every k_j

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads.  Window readings: "window 4096 (j in [i-4095, i])" is the
# causal window with max distance w = 4095; the Longformer workload is the
# symmetric window |i - j| <= 512 plus global tokens {0, 1000, 3000, 6000}.
TINY_FULL_F32 = Workload("tiny_full_f32_B1_H4_S256_d64", 1, 4, 4, 256, 64, "f32", MASK_FULL, seed=0)
CAUSAL_MHA_4K = Workload("causal_mha_B2_H32_S4096_d128", 2, 32, 32, 4096, 128, "bf16", MASK_CAUSAL,
                         seed=1, q_upper_heads_scale=2.0)
SWA_GQA_16K = Workload("causal_swa_gqa_B1_Hq32_Hkv8_S16384_d128_w4095", 1, 32, 8, 16384, 128, "bf16",
                       MASK_CAUSAL_SLIDING, window=4095, seed=2)
LONGFORMER_8K = Workload("local_global_B1_H12_S8192_d64_w512_g4", 1, 12, 12, 8192, 64, "bf16",
                         MASK_LOCAL_GLOBAL, window=512, globals_idx=(0, 1000, 3000, 6000), seed=3)
CAUSAL_GQA_32K = Workload("causal_gqa_B1_Hq64_Hkv8_S32768_d128", 1, 64, 8, 32768, 128, "bf16",
                          MASK_CAUSAL, seed=4, k_position_offset_std=0.5)

ALL = (TINY_FULL_F32, CAUSAL_MHA_4K, SWA_GQA_16K, LONGFORMER_8K, CAUSAL_GQA_32K)
BY_NAME = {w.name: w for w in ALL}


def make_inputs(w: Workload, device: Optional[str] = None):
    """Seeded Q [B,Hq,S,d], K, V [B,Hkv,S,d] in the workload dtype (CPU unless device given)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    Q = torch.randn(w.B, w.Hq, w.S, w.d, generator=g, dtype=torch.float32)
    K = torch.randn(w.B, w.Hkv, w.S, w.d, generator=g, dtype=torch.float32)
    V = torch.randn(w.B, w.Hkv, w.S, w.d, generator=g, dtype=torch.float32)
    if w.q_upper_heads_scale != 1.0:
        Q[:, w.Hq // 2:] *= w.q_upper_heads_scale
    if w.k_position_offset_std != 0.0:
        c = torch.randn(w.B, 1, w.S, 1, generator=g, dtype=torch.float32) * w.k_position_offset_std
        K += c
    Q, K, V = (t.to(w.torch_dtype) for t in (Q, K, V))
    if device is not None:
        Q, K, V = (t.to(device) for t in (Q, K, V))
    return Q, K, V


def allowed_pairs_per_head(w: Workload) -> int:
    """Closed-form count of allowed (i, j) pairs of one (batch, head) slice."""
    S, win = w.S, w.window

    def win_count(i):  # keys j with |i - j| <= win
        return min(i + win, S - 1) - max(i - win, 0) + 1

    if w.kind == MASK_FULL:
        return S * S
    if w.kind == MASK_CAUSAL:
        return S * (S + 1) // 2
    if w.kind == MASK_CAUSAL_SLIDING:
        return sum(min(i, win) + 1 for i in range(S))
    if w.kind == MASK_SLIDING:
        return sum(win_count(i) for i in range(S))
    # local + global: window pairs, plus the rest of each global row, plus each
    # global column's rows outside its window that are not themselves global
    G = sorted(set(w.globals_idx))
    total = sum(win_count(i) for i in range(S))
    total += sum(S - win_count(gi) for gi in G)
    for gj in G:
        outside = S - win_count(gj)
        outside -= sum(1 for gi in G if gi != gj and abs(gi - gj) > win)
        total += outside
    return total


def useful_flops(w: Workload) -> int:
    """4 * d flops per allowed pair (2d for the score, 2d for the weighted sum)."""
    return 4 * w.d * allowed_pairs_per_head(w) * w.B * w.Hq
