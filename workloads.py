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


# ----------------------------------------------------------------------------- decode
# Key/value-cache attention: S_q new query rows per sequence against a cache of
# capacity S_cap holding cache_len[b] positions of sequence b (ragged batch).
@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S_q: int
    S_cap: int
    d: int
    kind: int
    window: int = 0
    seed: int = 0
    len_min: int = 0        # cache lengths drawn uniformly from [len_min, S_cap]; 0 = all S_cap
    dtype: str = "bf16"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def with_(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)


# Long-context GQA decode (the 32K GQA head layout, one new token per sequence,
# eight sequences with ragged cache lengths in [16K, 32K]).
DECODE_GQA_32K = DecodeWorkload("decode_gqa_B8_Hq64_Hkv8_Sq1_cache32768_d128", 8, 64, 8, 1, 32768, 128,
                                MASK_CAUSAL, seed=10, len_min=16384)
# Four new positions per sequence (a chunk of prefill or of speculative tokens).
DECODE_GQA_CHUNK4 = DecodeWorkload("decode_gqa_B8_Hq32_Hkv8_Sq4_cache8192_d128", 8, 32, 8, 4, 8192, 128,
                                   MASK_CAUSAL, seed=11, len_min=1024)
# Multi-query decode: every query head shares one key/value head.
DECODE_MQA_16K = DecodeWorkload("decode_mqa_B16_Hq32_Hkv1_Sq1_cache16384_d128", 16, 32, 1, 1, 16384, 128,
                                MASK_CAUSAL, seed=12, len_min=2048)
# Sliding-window GQA decode (the window of the 16K sliding-window workload).
DECODE_SWA_16K = DecodeWorkload("decode_swa_B4_Hq32_Hkv8_Sq1_cache16384_d128_w4095", 4, 32, 8, 1, 16384, 128,
                                MASK_CAUSAL_SLIDING, window=4095, seed=13, len_min=4096)
# Cross-attention: 32 decoder rows against a 4096-position encoder output, d = 64.
CROSS_MHA_4K = DecodeWorkload("cross_mha_B4_H16_Sq32_enc4096_d64", 4, 16, 16, 32, 4096, 64, MASK_FULL,
                              seed=14)

DECODE_ALL = (DECODE_GQA_32K, DECODE_GQA_CHUNK4, DECODE_MQA_16K, DECODE_SWA_16K, CROSS_MHA_4K)
DECODE_BY_NAME = {w.name: w for w in DECODE_ALL}


def make_decode_inputs(w: DecodeWorkload, device: Optional[str] = None, stale_fill: float = 0.0):
    """Seeded Q [B,Hq,S_q,d], K, V [B,Hkv,S_cap,d] and cache lengths [B] (list of int).

    Draw order: Q, K, V (iid N(0, 1)), then the cache lengths.  Cache positions at
    or beyond a sequence's length are stale: they are set to ``stale_fill``
    (NaN in the tests, so that reading one shows up).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    Q = torch.randn(w.B, w.Hq, w.S_q, w.d, generator=g, dtype=torch.float32)
    K = torch.randn(w.B, w.Hkv, w.S_cap, w.d, generator=g, dtype=torch.float32)
    V = torch.randn(w.B, w.Hkv, w.S_cap, w.d, generator=g, dtype=torch.float32)
    if w.len_min > 0:
        lens = torch.randint(w.len_min, w.S_cap + 1, (w.B,), generator=g).tolist()
    else:
        lens = [w.S_cap] * w.B
    for b, L in enumerate(lens):
        K[b, :, L:] = stale_fill
        V[b, :, L:] = stale_fill
    Q, K, V = (t.to(w.torch_dtype) for t in (Q, K, V))
    if device is not None:
        Q, K, V = (t.to(device) for t in (Q, K, V))
    return Q, K, V, lens


def decode_keys_per_row(w: DecodeWorkload, L: int, i: int) -> int:
    """Closed-form count of the keys query row i sees in a sequence with L cached positions."""
    if w.kind == MASK_FULL:
        return L
    t = L - w.S_q + i
    if w.kind == MASK_CAUSAL:
        return t + 1
    return min(t, w.window) + 1  # causal sliding window


def decode_useful_flops(w: DecodeWorkload, lens) -> int:
    """4 * d flops per allowed (query row, key) pair."""
    pairs = sum(decode_keys_per_row(w, L, i) for L in lens for i in range(w.S_q))
    return 4 * w.d * pairs * w.Hq


def decode_bytes(w: DecodeWorkload, lens) -> int:
    """Algorithmic HBM bytes of one decode call: every key and value row some query of the
    group sees, read once per (sequence, kv head), plus Q and O (2 bytes) and LSE (4 bytes)."""
    el = 2 if w.dtype == "bf16" else 4
    kv_rows = 0
    for L in lens:
        if w.kind == MASK_CAUSAL_SLIDING:
            lo = max(0, L - w.S_q - w.window)
        else:
            lo = 0
        kv_rows += L - lo
    kv = 2 * kv_rows * w.Hkv * w.d * el
    qo = 2 * w.B * w.Hq * w.S_q * w.d * el
    return kv + qo + 4 * w.B * w.Hq * w.S_q


def alibi_slopes(H: int):
    """Slopes m_a = 2^(-8 (a + 1) / H) for H heads, a geometric sequence.  The pages fix one
    slope per head for the ALiBi bias -m_a |i - j| but give no values; this common choice
    is an input recipe, not something the pages state."""
    return [2.0 ** (-8.0 * (a + 1) / H) for a in range(H)]


def make_fp8_inputs(w: Workload):
    """E4M3 versions of the workload's Q, K, V with per-tensor descale factors.

    Each float32 tensor x of the recipe is scaled by 448 / max|x| (448: the largest finite
    E4M3 value), rounded to E4M3, and its descale is max|x| / 448.  Returns
    (Q8, K8, V8, (descale_q, descale_k, descale_v)) on the CPU.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    Q = torch.randn(w.B, w.Hq, w.S, w.d, generator=g, dtype=torch.float32)
    K = torch.randn(w.B, w.Hkv, w.S, w.d, generator=g, dtype=torch.float32)
    V = torch.randn(w.B, w.Hkv, w.S, w.d, generator=g, dtype=torch.float32)
    if w.q_upper_heads_scale != 1.0:
        Q[:, w.Hq // 2:] *= w.q_upper_heads_scale
    if w.k_position_offset_std != 0.0:
        K += torch.randn(w.B, 1, w.S, 1, generator=g, dtype=torch.float32) * w.k_position_offset_std
    out, ds = [], []
    for x in (Q, K, V):
        amax = float(x.abs().max())
        out.append((x * (448.0 / amax)).to(torch.float8_e4m3fn))
        ds.append(amax / 448.0)
    return out[0], out[1], out[2], tuple(ds)


# ----------------------------------------------------------------------------- backward
def make_grad_output(w: Workload, device: Optional[str] = None):
    """Seeded output gradient dO [B, Hq, S, d] in the workload dtype: standard normal entries,
    drawn from a generator seeded with seed + 1 so it is independent of Q, K and V."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 1)
    dO = torch.randn(w.B, w.Hq, w.S, w.d, generator=g, dtype=torch.float32).to(w.torch_dtype)
    return dO if device is None else dO.to(device)


def backward_flops(w: Workload) -> int:
    """10 * d flops per allowed pair: the backward's five products of the (query, key) pair
    (the score and dP, and the dQ, dK and dV updates), 2d flops each.  2.5 times the forward."""
    return 10 * w.d * allowed_pairs_per_head(w) * w.B * w.Hq
