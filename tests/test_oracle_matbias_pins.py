"""Pins of the oracle's general additive bias matrix: logits_ij = scale * q_i . k_j + b_ij
with b given as a tensor [Bb, Hb, S, ld] ("Transformer 架构及其变体", the unified
biased-logits form, where b_ij is any bias added to the scaled scores).  No GPU.
"""
import numpy as np
import pytest
import torch

import oracle

KINDS = (oracle.MASK_FULL, oracle.MASK_CAUSAL, oracle.MASK_SLIDING, oracle.MASK_CAUSAL_SLIDING,
         oracle.MASK_LOCAL_GLOBAL)


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def _torch_ref(Q, K, V, scale, kind, w, G, bias):
    """float64 torch.softmax over the logits with the bias added element by element."""
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    Bb, Hb = bias.shape[:2]
    M = torch.zeros(S, S, dtype=torch.bool)
    for i in range(S):
        for j in range(S):
            M[i, j] = oracle.allowed(kind, i, j, S, w, G)
    O = torch.empty(B, Hq, S, d, dtype=torch.float64)
    L = torch.empty(B, Hq, S, dtype=torch.float64)
    for b in range(B):
        for a in range(Hq):
            g = a // (Hq // Hkv)
            s = torch.from_numpy(Q[b, a]).double() @ torch.from_numpy(K[b, g]).double().T * scale
            s = s + torch.from_numpy(bias[0 if Bb == 1 else b, 0 if Hb == 1 else a, :, :S]).double()
            s = s.masked_fill(~M, float("-inf"))
            O[b, a] = torch.softmax(s, -1) @ torch.from_numpy(V[b, g]).double()
            L[b, a] = torch.logsumexp(s, -1)
    return O.numpy(), L.numpy()


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("Bb,Hb", [(1, 1), (2, 1), (1, 4), (2, 4)])
def test_bias_matrix_matches_library_softmax(kind, Bb, Hb):
    B, Hq, Hkv, S, d = 2, 4, 2, 29, 8
    Q, K, V = _rand((B, Hq, S, d), 1), _rand((B, Hkv, S, d), 2), _rand((B, Hkv, S, d), 3)
    bias = _rand((Bb, Hb, S, 32), 4, 1.5)  # row stride 32 > S
    G = [0, 17] if kind == oracle.MASK_LOCAL_GLOBAL else None
    O, L = oracle.attention(Q, K, V, 0.35, kind, 5, G, bias=bias)
    O_t, L_t = _torch_ref(Q, K, V, 0.35, kind, 5, G, bias)
    assert np.allclose(O, O_t, atol=1e-12, rtol=0) and np.allclose(L, L_t, atol=1e-12, rtol=0)


@pytest.mark.parametrize("kind", KINDS)
def test_alibi_distance_matrix_is_the_alibi_bias(kind):
    """b_ij = -m_a |i - j| written out as a [1, Hq, S, S] matrix gives the (pinned) ALiBi result."""
    B, Hq, S, d = 1, 3, 21, 4
    Q, K, V = _rand((B, Hq, S, d), 5), _rand((B, Hq, S, d), 6), _rand((B, Hq, S, d), 7)
    slopes = [0.5, 0.125, 2.0]
    dist = np.abs(np.arange(S)[:, None] - np.arange(S)[None, :]).astype(np.float64)
    bias = np.stack([-m * dist for m in slopes])[None].astype(np.float32)
    G = [3] if kind == oracle.MASK_LOCAL_GLOBAL else None
    a = oracle.attention(Q, K, V, 0.4, kind, 4, G, alibi=slopes)
    b = oracle.attention(Q, K, V, 0.4, kind, 4, G, bias=bias)
    assert np.allclose(a[0], b[0], atol=1e-12) and np.allclose(a[1], b[1], atol=1e-12)


@pytest.mark.parametrize("kind", KINDS)
def test_row_constant_bias_shifts_only_the_lse(kind):
    """Softmax is shift invariant: b_ij = c_i leaves O and moves LSE_i by c_i."""
    B, Hq, S, d = 2, 2, 19, 4
    Q, K, V = _rand((B, Hq, S, d), 8), _rand((B, Hq, S, d), 9), _rand((B, Hq, S, d), 10)
    c = _rand((B, Hq, S), 11, 3.0)
    bias = np.repeat(c[..., None], S, axis=3)
    G = [0, 9] if kind == oracle.MASK_LOCAL_GLOBAL else None
    O0, L0 = oracle.attention(Q, K, V, 0.5, kind, 3, G)
    O1, L1 = oracle.attention(Q, K, V, 0.5, kind, 3, G, bias=bias)
    assert np.allclose(O0, O1, atol=1e-12) and np.allclose(L1, L0 + c, atol=1e-11)


def test_padding_columns_are_never_read():
    """Row-stride padding (ld > S) filled with NaN changes nothing."""
    B, Hq, S, d = 1, 2, 13, 4
    Q, K, V = _rand((B, Hq, S, d), 12), _rand((B, Hq, S, d), 13), _rand((B, Hq, S, d), 14)
    bias = _rand((1, Hq, S, 16), 15)
    padded = bias.copy()
    padded[..., S:] = np.nan
    a = oracle.attention(Q, K, V, 0.5, oracle.MASK_FULL, bias=bias)
    b = oracle.attention(Q, K, V, 0.5, oracle.MASK_FULL, bias=padded)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_minus_infinity_above_the_diagonal_is_the_causal_mask():
    B, Hq, S, d = 1, 2, 17, 4
    Q, K, V = _rand((B, Hq, S, d), 16), _rand((B, Hq, S, d), 17), _rand((B, Hq, S, d), 18)
    tri = np.where(np.arange(S)[None, :] > np.arange(S)[:, None], -np.inf, 0.0).astype(np.float32)
    a = oracle.attention(Q, K, V, 0.5, oracle.MASK_CAUSAL)
    b = oracle.attention(Q, K, V, 0.5, oracle.MASK_FULL, bias=tri[None, None])
    assert np.allclose(a[0], b[0], atol=1e-13) and np.allclose(a[1], b[1], atol=1e-13)
