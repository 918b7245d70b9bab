"""The multi-GPU split of one problem (whole kv-head groups per rank) and the bench's
max-over-ranks timing, on world-size-2 gloo process groups on the CPU.

Each rank computes its share with the oracle (the attention kernels need a GPU); the test
is that the shares cover every head once, that the all-gather rebuilds exactly the oracle's
result for the whole problem (uneven shares and an empty share included), and that every
rank sees the slowest rank's time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from transformer_self_attention_gb300.shard import gather_heads, kv_head_range, max_over_ranks, shard_heads

CASES = [(2, 6, 3, 70, 8, 1), (1, 4, 1, 33, 4, 0), (2, 8, 4, 40, 4, 3)]  # B, Hq, Hkv, S, d, kind


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(B, Hq, Hkv, S, d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, Hq, S, d, generator=g), torch.randn(B, Hkv, S, d, generator=g),
            torch.randn(B, Hkv, S, d, generator=g))


def _worker(rank, world, port):
    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        for seed, (B, Hq, Hkv, S, d, kind) in enumerate(CASES):
            Q, K, V = _inputs(B, Hq, Hkv, S, d, seed)
            q, k, v = shard_heads(Q, K, V, world, rank)
            if q.shape[1]:
                O, L = oracle.attention(q.numpy(), k.numpy(), v.numpy(), 0.3, kind, 5)
                O, L = torch.from_numpy(O), torch.from_numpy(L)
            else:  # this rank holds no kv head
                O, L = torch.zeros(B, 0, S, d, dtype=torch.float64), torch.zeros(B, 0, S, dtype=torch.float64)
            O_all, L_all = gather_heads(O, L, Hq, Hkv)
            O_ref, L_ref = oracle.attention(Q.numpy(), K.numpy(), V.numpy(), 0.3, kind, 5)
            assert np.array_equal(O_all.numpy(), O_ref) and np.array_equal(L_all.numpy(), L_ref), (rank, seed)
        assert max_over_ranks(10.0 * rank + 1.0) == 10.0 * (world - 1) + 1.0
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_split_over_two_ranks_rebuilds_the_whole_result():
    mp.spawn(_worker, args=(2, _free_port()), nprocs=2, join=True)


@pytest.mark.parametrize("Hkv", [1, 2, 3, 8, 13])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_kv_head_ranges_cover_every_head_once(Hkv, world):
    ranges = [kv_head_range(Hkv, world, r) for r in range(world)]
    heads = [g for lo, hi in ranges for g in range(lo, hi)]
    assert heads == list(range(Hkv))
    sizes = [hi - lo for lo, hi in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_max_over_ranks_without_a_process_group():
    assert max_over_ranks(3.5) == 3.5
