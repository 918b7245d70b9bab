"""One attention problem over several GPUs: whole key/value-head groups per rank.

Every (batch, kv head) unit -- its K and V and the query heads that share them -- is
independent of the others (the grouped-query sharing of "Transformer 演进与变体"
(ai.icyfenix.cn), section GQA：分组查询注意力: query heads a with g(a) = a / (Hq / Hkv) read
kv head g only).  So the heads split over ranks with no exchange step: rank r takes the
kv heads [g0, g1) and their query heads [g0 * group, g1 * group), computes them alone, and
an all-gather over heads rebuilds O and LSE only where one rank needs the whole output.

This module holds the index arithmetic and the torch.distributed plumbing; the attention
itself runs in the library's kernels on each rank's GPU.
"""
from __future__ import annotations


def kv_head_range(Hkv: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced share [g0, g1) of the Hkv kv heads for `rank` of `world` ranks
    (sizes differ by at most one; ranks beyond Hkv get an empty range)."""
    if world < 1 or not 0 <= rank < world or Hkv < 1:
        raise ValueError("need Hkv >= 1 and 0 <= rank < world")
    return rank * Hkv // world, (rank + 1) * Hkv // world


def shard_heads(Q, K, V, world: int, rank: int):
    """This rank's slices of Q [B, Hq, S, d] and K, V [B, Hkv, S, d]: the kv heads of
    kv_head_range and their query heads, as contiguous tensors."""
    Hq, Hkv = Q.shape[1], K.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    g0, g1 = kv_head_range(Hkv, world, rank)
    return (Q[:, g0 * group:g1 * group].contiguous(), K[:, g0:g1].contiguous(), V[:, g0:g1].contiguous())


def gather_heads(O_local, LSE_local, Hq: int, Hkv: int, group=None):
    """All-gather of every rank's O [B, hq_r, S, d] and LSE [B, hq_r, S] into the full
    O [B, Hq, S, d] and LSE [B, Hq, S] on every rank (shares padded to the largest for the
    collective, then trimmed).  `group`: a torch.distributed process group (default: world)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    per = Hq // Hkv
    sizes = [(kv_head_range(Hkv, world, r)[1] - kv_head_range(Hkv, world, r)[0]) * per for r in range(world)]
    mx = max(sizes)
    B, h, S = O_local.shape[0], O_local.shape[1], O_local.shape[2]
    d = O_local.shape[3]
    pad_o = O_local.new_zeros((B, mx, S, d))
    pad_l = LSE_local.new_zeros((B, mx, S))
    pad_o[:, :h] = O_local
    pad_l[:, :h] = LSE_local
    outs_o = [torch.empty_like(pad_o) for _ in range(world)]
    outs_l = [torch.empty_like(pad_l) for _ in range(world)]
    dist.all_gather(outs_o, pad_o, group=group)
    dist.all_gather(outs_l, pad_l, group=group)
    O = torch.cat([o[:, :n] for o, n in zip(outs_o, sizes)], dim=1)
    LSE = torch.cat([l[:, :n] for l, n in zip(outs_l, sizes)], dim=1)
    return O, LSE


def max_over_ranks(value: float, device=None, group=None) -> float:
    """The largest `value` over all ranks (the slowest rank's time); `value` when not distributed."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized():
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
