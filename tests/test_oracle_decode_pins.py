"""Pins of the fp64 decode (key/value-cache) oracle.

The decode form follows "Trasformer 浅析" (sections 推理：KV 缓存 and 交叉注意力)
and "第 8 章 现代大模型架构" (section 预填充创建缓存，解码复用缓存).  Each test
would catch a plausible mistake: the new rows placed one position off, stale
cache entries read, the window off by one, a wrong g(a), a missing scale or
normalisation.  No GPU.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

DEC_KINDS = (oracle.MASK_FULL, oracle.MASK_CAUSAL, oracle.MASK_CAUSAL_SLIDING)


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(np.float32)


@pytest.mark.parametrize("kind,w", [(oracle.MASK_CAUSAL, 0), (oracle.MASK_CAUSAL_SLIDING, 3),
                                    (oracle.MASK_CAUSAL_SLIDING, 0), (oracle.MASK_FULL, 0)])
@pytest.mark.parametrize("S_q", [1, 3, 7])
def test_decode_rows_are_the_last_rows_of_prefill(kind, w, S_q):
    """Decoding the last S_q positions of a full cache gives the same rows as the square
    (prefill) oracle over the whole sequence: cached keys and values do not change, so the
    step-t output is row t of the masked self-attention (KV-cache section)."""
    B, Hq, Hkv, S, d = 2, 4, 2, 19, 8
    Qf = _rand((B, Hq, S, d), 1)
    K = _rand((B, Hkv, S, d), 2)
    V = _rand((B, Hkv, S, d), 3)
    scale = 1 / math.sqrt(d)
    O_ref, L_ref = oracle.attention(Qf, K, V, scale, kind, w)
    O, LSE = oracle.decode(Qf[:, :, S - S_q:], K, V, [S] * B, scale, kind, w)
    assert np.allclose(O, O_ref[:, :, S - S_q:], atol=1e-13, rtol=0)
    assert np.allclose(LSE, L_ref[:, :, S - S_q:], atol=1e-13, rtol=0)


@pytest.mark.parametrize("kind,w", [(oracle.MASK_CAUSAL, 0), (oracle.MASK_CAUSAL_SLIDING, 5),
                                    (oracle.MASK_FULL, 0)])
def test_decode_ragged_batch_ignores_stale_cache(kind, w):
    """A ragged batch (sequence r holds S_r cached positions): sequence b equals the prefill
    oracle on its own first cache_len[b] positions, and NaN in the stale part of the cache
    never reaches the output."""
    B, Hq, Hkv, S_cap, d, S_q = 3, 4, 1, 48, 8, 2
    lens = [5, 17, 48]
    Qf = _rand((B, Hq, S_cap, d), 4)
    K = _rand((B, Hkv, S_cap, d), 5)
    V = _rand((B, Hkv, S_cap, d), 6)
    Kp, Vp, Q = K.copy(), V.copy(), np.empty((B, Hq, S_q, d), np.float32)
    for b, L in enumerate(lens):
        Kp[b, :, L:] = np.nan
        Vp[b, :, L:] = np.nan
        Q[b] = Qf[b, :, L - S_q:L]
    O, LSE = oracle.decode(Q, Kp, Vp, lens, 0.3, kind, w)
    assert np.isfinite(O).all() and np.isfinite(LSE).all()
    for b, L in enumerate(lens):
        O_ref, L_ref = oracle.attention(Qf[b:b + 1, :, :L], K[b:b + 1, :, :L], V[b:b + 1, :, :L], 0.3, kind, w)
        assert np.allclose(O[b], O_ref[0, :, L - S_q:], atol=1e-13, rtol=0)
        assert np.allclose(LSE[b], L_ref[0, :, L - S_q:], atol=1e-13, rtol=0)


@pytest.mark.parametrize("kind", DEC_KINDS)
def test_decode_first_token(kind):
    """A cache holding one position: the only key is the query's own, so O = v_0 and
    LSE = scale * q . k_0 (the first row of the causal mask sees only itself)."""
    d = 5
    Q = _rand((1, 3, 1, d), 7)
    K = _rand((1, 1, 4, d), 8)
    V = _rand((1, 1, 4, d), 9)
    O, LSE = oracle.decode(Q, K, V, [1], 0.7, kind, 2)
    for a in range(3):
        assert np.allclose(O[0, a, 0], V[0, 0, 0], atol=1e-15)
        assert LSE[0, a, 0] == pytest.approx(0.7 * float(np.dot(Q[0, a, 0].astype(np.float64),
                                                               K[0, 0, 0].astype(np.float64))), abs=1e-13)


def test_cross_attention_matches_library_softmax():
    """Cross-attention (an n_dec x n_enc score matrix, every encoder key visible) equals
    float64 torch.softmax(Q_dec K_enc^T * scale) @ V_enc."""
    B, H, n_dec, n_enc, d = 2, 3, 7, 13, 6
    Q = _rand((B, H, n_dec, d), 10)
    K = _rand((B, H, n_enc, d), 11)
    V = _rand((B, H, n_enc, d), 12)
    scale = 1 / math.sqrt(d)
    O, LSE = oracle.decode(Q, K, V, [n_enc] * B, scale, oracle.MASK_FULL)
    q, k, v = (torch.from_numpy(x).double() for x in (Q, K, V))
    s = q @ k.transpose(-1, -2) * scale
    ref = torch.softmax(s, dim=-1) @ v
    assert np.allclose(O, ref.numpy(), atol=1e-13, rtol=0)
    assert np.allclose(LSE, torch.logsumexp(s, dim=-1).numpy(), atol=1e-13, rtol=0)


@pytest.mark.parametrize("kind", DEC_KINDS)
def test_decode_gqa_equals_repeated_kv_heads(kind):
    """Grouped heads: Hq query heads over Hkv cached heads equal MHA with every cached head
    repeated for the Hq/Hkv query heads of its group (g(a) = a // (Hq/Hkv))."""
    B, Hq, Hkv, S_q, S_cap, d = 2, 6, 2, 3, 20, 4
    Q = _rand((B, Hq, S_q, d), 13)
    K = _rand((B, Hkv, S_cap, d), 14)
    V = _rand((B, Hkv, S_cap, d), 15)
    lens = [11, 20]
    O, LSE = oracle.decode(Q, K, V, lens, 0.5, kind, 4)
    Kr, Vr = np.repeat(K, Hq // Hkv, axis=1), np.repeat(V, Hq // Hkv, axis=1)
    O2, LSE2 = oracle.decode(Q, Kr, Vr, lens, 0.5, kind, 4)
    assert np.array_equal(O, O2) and np.array_equal(LSE, LSE2)
    # and a wrong grouping (interleaved heads) would differ
    Ki, Vi = np.tile(K, (1, Hq // Hkv, 1, 1)), np.tile(V, (1, Hq // Hkv, 1, 1))
    O3, _ = oracle.decode(Q, Ki, Vi, lens, 0.5, kind, 4)
    assert not np.allclose(O, O3)


@pytest.mark.parametrize("w", [0, 1, 3, 6])
def test_decode_window_support(w):
    """With V = I the output row is the weight vector; its support must be exactly the keys
    j with t - w <= j <= t (t the row's position), and the weights the softmax of the
    scaled scores on that support."""
    L, S_q, d = 12, 3, 12
    Q = _rand((1, 1, S_q, d), 16)
    K = _rand((1, 1, L, d), 17)
    V = np.eye(L, dtype=np.float32)[None, None]
    O, _ = oracle.decode(Q, K, V, [L], 0.4, oracle.MASK_CAUSAL_SLIDING, w)
    for i in range(S_q):
        t = L - S_q + i
        support = [j for j in range(L) if O[0, 0, i, j] > 0]
        assert support == list(range(max(0, t - w), t + 1))
        s = 0.4 * (K[0, 0, support].astype(np.float64) @ Q[0, 0, i].astype(np.float64))
        e = np.exp(s - s.max())
        assert np.allclose(O[0, 0, i, support], e / e.sum(), atol=1e-14)


def test_decode_predicate_examples():
    """The decode predicate at the pages' window example (w = 3, a query at position 5 sees
    positions 2..5 once the future is cut off) and at the cache edge."""
    L = 9
    assert [j for j in range(L) if oracle.decode_allowed(oracle.MASK_CAUSAL_SLIDING, 5, j, L, 3)] == [2, 3, 4, 5]
    assert [j for j in range(L) if oracle.decode_allowed(oracle.MASK_CAUSAL, 5, j, L)] == list(range(6))
    assert [j for j in range(L + 3) if oracle.decode_allowed(oracle.MASK_FULL, 0, j, L)] == list(range(L))
    assert not oracle.decode_allowed(oracle.MASK_SLIDING, 5, 5, L, 3)  # not a decode kind


def test_decode_constant_values_and_unit_rows():
    """Rows of the attention matrix sum to one: V constant over positions returns the
    constant, for every decode kind and ragged lengths."""
    B, Hq, Hkv, S_q, S_cap, d = 2, 4, 2, 2, 30, 3
    Q = _rand((B, Hq, S_q, d), 18, 3.0)
    K = _rand((B, Hkv, S_cap, d), 19)
    c = np.array([1.5, -2.0, 0.25], dtype=np.float32)
    V = np.broadcast_to(c, (B, Hkv, S_cap, d)).copy()
    for kind in DEC_KINDS:
        O, _ = oracle.decode(Q, K, V, [7, 30], 1.0, kind, 2)
        assert np.allclose(O, np.broadcast_to(c, O.shape), atol=1e-14)


def test_decode_rejects_bad_lengths():
    Q = _rand((1, 1, 4, 2), 20)
    K = _rand((1, 1, 8, 2), 21)
    with pytest.raises(ValueError):
        oracle.decode(Q, K, K, [3], 1.0, oracle.MASK_CAUSAL)      # fewer cached positions than new rows
    with pytest.raises(ValueError):
        oracle.decode(Q, K, K, [9], 1.0, oracle.MASK_CAUSAL)      # beyond the capacity
    with pytest.raises(ValueError):
        oracle.decode(Q, K, K, [8], 1.0, oracle.MASK_SLIDING)     # not a decode kind
    O, _ = oracle.decode(Q, K, K, [2], 1.0, oracle.MASK_FULL)     # cross-attention: any length >= 1
    assert O.shape == (1, 1, 4, 2)


def test_decode_workload_counts():
    """The closed-form key counts of the decode workloads agree with enumeration of the
    oracle's predicate on small lengths."""
    for w in wl.DECODE_ALL:
        small = w.with_(window=min(w.window, 37))
        for L in (small.S_q, small.S_q + 1, 40, 129):
            for i in range(small.S_q):
                t = L - small.S_q + i
                n = sum(oracle.decode_allowed(small.kind, t, j, L, small.window) for j in range(L))
                assert n == wl.decode_keys_per_row(small, L, i), (w.name, L, i)
