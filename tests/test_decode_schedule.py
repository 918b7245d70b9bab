"""The decode chunking (host only) against brute force from the oracle's decode predicate.

The key tiles a CTA streams are derived from (tiles_per_chunk, chunk_prefix) exactly
as the kernel derives them; the chunks of every sequence must cover its key-tile
range once, in order and without empty chunks, and that range must hold every key
some query row of the sequence is allowed to see (and begin at the first tile
holding one).  Bit-exact; no GPU.
"""
import random

import numpy as np
import pytest

import oracle
import transformer_self_attention_gb300 as tsa

T = tsa.TILE
KINDS = (tsa.MASK_FULL, tsa.MASK_CAUSAL, tsa.MASK_CAUSAL_SLIDING)


def _kernel_chunks(tpc, prefix, b, kind, S_q, window, L):
    """The key tiles of each chunk of sequence b, as the kernel computes them."""
    t_lo = max(0, L - S_q - window) // T if kind == tsa.MASK_CAUSAL_SLIDING else 0
    t_hi = (L + T - 1) // T
    out = []
    for c in range(prefix[b + 1] - prefix[b]):
        t0 = t_lo + c * tpc
        n = min(t_hi, t0 + tpc) - t0
        out.append((t0, t0 + n))
    return out


def _needed_tiles(kind, S_q, window, L):
    """Key tiles holding at least one key some row may see (brute force over the predicate)."""
    tiles = set()
    for i in range(S_q):
        t = L - S_q + i
        for j in range(L):
            if oracle.decode_allowed(kind, t, j, L, window):
                tiles.add(j // T)
    return tiles


def _check(B, Hkv, S_q, S_cap, kind, window, lens, n_sm):
    tpc, prefix = tsa.attn_decode_schedule_host(B, Hkv, S_q, S_cap, kind, window, lens, n_sm)
    assert tpc >= 1 and prefix[0] == 0
    for b, L in enumerate(lens):
        chunks = _kernel_chunks(tpc, prefix, b, kind, S_q, window, L)
        assert 1 <= len(chunks) <= 256
        assert all(e > s for s, e in chunks), "empty chunk"
        assert all(chunks[k][1] == chunks[k + 1][0] for k in range(len(chunks) - 1))
        covered = set(range(chunks[0][0], chunks[-1][1]))
        need = _needed_tiles(kind, S_q, window, L)
        assert need <= covered
        assert min(covered) == min(need) and max(covered) == max(need)
    n_cta = int(prefix[-1]) * Hkv
    assert n_cta <= n_sm + B * Hkv
    return tpc, prefix


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("S_q", [1, 2, 5])
def test_decode_chunks_cover_the_allowed_keys(kind, S_q):
    rng = random.Random(kind * 10 + S_q)
    for trial in range(6):
        B = rng.randint(1, 5)
        Hkv = rng.choice([1, 2, 8])
        S_cap = rng.choice([S_q, 127, 128, 129, 300, 1000])
        S_cap = max(S_cap, S_q)
        lens = [rng.randint(S_q if kind != tsa.MASK_FULL else 1, S_cap) for _ in range(B)]
        window = rng.choice([0, 1, 127, 128, 200])
        _check(B, Hkv, S_q, S_cap, kind, window, lens, n_sm=rng.choice([1, 7, 152]))


def test_decode_chunks_fill_the_gpu_for_long_caches():
    """Eight long sequences with 8 kv heads: chunks sized so the launch is about one CTA per SM."""
    lens = [16384 + 2000 * b for b in range(8)]
    tpc, prefix = tsa.attn_decode_schedule_host(8, 8, 1, 32768, tsa.MASK_CAUSAL, 0, lens, 152)
    n_cta = int(prefix[-1]) * 8
    assert 152 <= n_cta <= 152 + 64
    total_tiles = sum((L + T - 1) // T for L in lens) * 8
    assert tpc == -(-total_tiles // 152)


def test_decode_chunk_cap_per_sequence():
    """A single very long sequence on a large GPU is not split into more than 256 chunks."""
    tpc, prefix = tsa.attn_decode_schedule_host(1, 1, 1, 1 << 20, tsa.MASK_CAUSAL, 0, [1 << 20], 100000)
    assert prefix[1] <= 256 and tpc * prefix[1] >= (1 << 20) // T


def test_decode_sliding_window_skips_old_tiles():
    """The causal window reads only the tiles of the last window + S_q positions."""
    L, w = 16384, 4095
    tpc, prefix = tsa.attn_decode_schedule_host(1, 8, 1, L, tsa.MASK_CAUSAL_SLIDING, w, [L], 152)
    chunks = _kernel_chunks(tpc, prefix, 0, tsa.MASK_CAUSAL_SLIDING, 1, w, L)
    assert chunks[0][0] == (L - 1 - w) // T and chunks[-1][1] == L // T


@pytest.mark.parametrize("args,status", [
    ((1, 1, 1, 8, tsa.MASK_SLIDING, 2, [8], 4), tsa.ATTN_ERR_UNSUPPORTED),       # not a decode kind
    ((1, 1, 1, 8, tsa.MASK_LOCAL_GLOBAL, 2, [8], 4), tsa.ATTN_ERR_UNSUPPORTED),
    ((1, 1, 65, 100, tsa.MASK_CAUSAL, 0, [100], 4), tsa.ATTN_ERR_UNSUPPORTED),   # more than 64 rows
    ((1, 1, 4, 8, tsa.MASK_CAUSAL, 0, [3], 4), tsa.ATTN_ERR_INVALID_ARG),        # fewer cached than new rows
    ((1, 1, 1, 8, tsa.MASK_CAUSAL, 0, [9], 4), tsa.ATTN_ERR_INVALID_ARG),        # beyond the capacity
    ((1, 1, 1, 8, tsa.MASK_CAUSAL, 0, [0], 4), tsa.ATTN_ERR_INVALID_ARG),        # empty cache
    ((1, 1, 1, 8, tsa.MASK_CAUSAL_SLIDING, -1, [8], 4), tsa.ATTN_ERR_INVALID_ARG),
    ((1, 1, 1, 8, tsa.MASK_CAUSAL, 0, [8], 0), tsa.ATTN_ERR_INVALID_ARG),        # no multiprocessor
    ((1025, 1, 1, 8, tsa.MASK_CAUSAL, 0, [8] * 1025, 4), tsa.ATTN_ERR_UNSUPPORTED),
])
def test_decode_schedule_validation(args, status):
    with pytest.raises(tsa.AttnError) as e:
        tsa.attn_decode_schedule_host(*args)
    assert e.value.status == status


def test_cross_attention_lengths_may_be_shorter_than_the_query_rows():
    tpc, prefix = tsa.attn_decode_schedule_host(2, 4, 32, 4096, tsa.MASK_FULL, 0, [3, 4096], 152)
    assert prefix[1] == 1


@pytest.mark.parametrize("kw,status", [
    (dict(B=1, Hq=4, Hkv=4, S_q=1, S_cap=64, d_k=96, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_UNSUPPORTED),
    (dict(B=1, Hq=4, Hkv=4, S_q=1, S_cap=64, d_k=64, scale=0.0, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_INVALID_ARG),
    (dict(B=1, Hq=4, Hkv=3, S_q=1, S_cap=64, d_k=64, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_INVALID_ARG),
    (dict(B=1, Hq=64, Hkv=1, S_q=2, S_cap=64, d_k=64, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_UNSUPPORTED),
    (dict(B=1, Hq=4, Hkv=4, S_q=8, S_cap=4, d_k=64, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_INVALID_ARG),
    (dict(B=1, Hq=4, Hkv=4, S_q=1, S_cap=64, d_k=64, scale=0.1, kind=tsa.MASK_SLIDING), tsa.ATTN_ERR_UNSUPPORTED),
])
def test_decode_create_rejects_bad_arguments_before_any_cuda_call(kw, status):
    with pytest.raises(tsa.AttnError) as e:
        tsa.attn_decode_create(**kw)
    assert e.value.status == status
