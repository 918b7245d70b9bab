"""Pins of the oracle's additive score bias (ALiBi): logits_ij = scale * q_i . k_j + b_ij with
b_ij = -m_a |i - j| ("Transformer 架构及其变体", the unified biased-logits form and section
加性偏置：ALiBi; "Trasformer 浅析", section 线性偏置注意力).  No GPU.
"""
import math

import numpy as np
import pytest
import torch

import oracle

KINDS = (oracle.MASK_FULL, oracle.MASK_CAUSAL, oracle.MASK_SLIDING, oracle.MASK_CAUSAL_SLIDING,
         oracle.MASK_LOCAL_GLOBAL)


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def _allowed_matrix(kind, S, w, G):
    M = np.zeros((S, S), dtype=bool)
    for i in range(S):
        for j in range(S):
            M[i, j] = oracle.allowed(kind, i, j, S, w, G)
    return M


def _torch_ref(Q, K, V, scale, kind, w, G, slopes, signed_causal=False):
    """float64 torch.softmax over logits with the bias matrix written out element by element."""
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    M = torch.from_numpy(_allowed_matrix(kind, S, w, G))
    i = torch.arange(S)[:, None].double()
    j = torch.arange(S)[None, :].double()
    dist = (i - j) if signed_causal else (i - j).abs()
    O = torch.empty(B, Hq, S, d, dtype=torch.float64)
    L = torch.empty(B, Hq, S, dtype=torch.float64)
    for b in range(B):
        for a in range(Hq):
            g = a // (Hq // Hkv)
            s = torch.from_numpy(Q[b, a]).double() @ torch.from_numpy(K[b, g]).double().T * scale
            s = s - float(slopes[a]) * dist
            s = s.masked_fill(~M, float("-inf"))
            O[b, a] = torch.softmax(s, -1) @ torch.from_numpy(V[b, g]).double()
            L[b, a] = torch.logsumexp(s, -1)
    return O.numpy(), L.numpy()


@pytest.mark.parametrize("kind", KINDS)
def test_alibi_matches_library_softmax(kind):
    B, Hq, Hkv, S, d = 1, 4, 2, 37, 8
    Q, K, V = _rand((B, Hq, S, d), 1), _rand((B, Hkv, S, d), 2), _rand((B, Hkv, S, d), 3)
    slopes = [0.5, 0.25, 0.125, 0.0625]
    G = [0, 20] if kind == oracle.MASK_LOCAL_GLOBAL else None
    O, L = oracle.attention(Q, K, V, 0.35, kind, 5, G, alibi=slopes)
    O_t, L_t = _torch_ref(Q, K, V, 0.35, kind, 5, G, slopes)
    assert np.allclose(O, O_t, atol=1e-12, rtol=0) and np.allclose(L, L_t, atol=1e-12, rtol=0)


def test_causal_signed_distance_form_is_the_same():
    """-m (i - j) for j <= i (the causal form) and -m |i - j| give the same causal attention."""
    B, Hq, S, d = 1, 2, 29, 4
    Q, K, V = _rand((B, Hq, S, d), 4), _rand((B, Hq, S, d), 5), _rand((B, Hq, S, d), 6)
    O, L = oracle.attention(Q, K, V, 0.5, oracle.MASK_CAUSAL, alibi=[0.3, 0.7])
    O_t, L_t = _torch_ref(Q, K, V, 0.5, oracle.MASK_CAUSAL, 0, None, [0.3, 0.7], signed_causal=True)
    assert np.allclose(O, O_t, atol=1e-12, rtol=0) and np.allclose(L, L_t, atol=1e-12, rtol=0)


@pytest.mark.parametrize("kind", KINDS)
def test_zero_slopes_are_no_bias(kind):
    B, Hq, S, d = 2, 2, 23, 4
    Q, K, V = _rand((B, Hq, S, d), 7), _rand((B, Hq, S, d), 8), _rand((B, Hq, S, d), 9)
    G = [3] if kind == oracle.MASK_LOCAL_GLOBAL else None
    a = oracle.attention(Q, K, V, 0.4, kind, 3, G)
    b = oracle.attention(Q, K, V, 0.4, kind, 3, G, alibi=[0.0, 0.0])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("kind", KINDS)
def test_steep_slope_keeps_only_the_own_position(kind):
    """Every row sees itself with zero bias and every other key with at least -m: a steep slope
    leaves O_i = v_i and LSE_i = scale * q_i . k_i."""
    B, Hq, S, d = 1, 2, 19, 4
    Q, K, V = _rand((B, Hq, S, d), 10), _rand((B, Hq, S, d), 11), _rand((B, Hq, S, d), 12)
    G = [0, 9] if kind == oracle.MASK_LOCAL_GLOBAL else None
    O, L = oracle.attention(Q, K, V, 0.5, kind, 4, G, alibi=[200.0, 200.0])
    assert np.allclose(O, V.astype(np.float64), atol=1e-12)
    diag = 0.5 * np.einsum("bhid,bhid->bhi", Q.astype(np.float64), K.astype(np.float64))
    assert np.allclose(L, diag, atol=1e-12)


def test_slope_belongs_to_the_query_head():
    """Query heads of one kv group with different slopes: head a uses slope a."""
    B, Hq, Hkv, S, d = 1, 4, 1, 21, 4
    Q, K, V = _rand((B, Hq, S, d), 13), _rand((B, Hkv, S, d), 14), _rand((B, Hkv, S, d), 15)
    slopes = [0.0, 0.1, 1.0, 3.0]
    O, _ = oracle.attention(Q, K, V, 0.5, oracle.MASK_CAUSAL, alibi=slopes)
    for a in range(Hq):
        Oa, _ = oracle.attention(Q[:, a:a + 1], K, V, 0.5, oracle.MASK_CAUSAL, alibi=[slopes[a]])
        assert np.array_equal(O[:, a:a + 1], Oa)


@pytest.mark.parametrize("kind,w", [(oracle.MASK_CAUSAL, 0), (oracle.MASK_CAUSAL_SLIDING, 4), (oracle.MASK_FULL, 0)])
def test_decode_bias_is_the_prefill_bias_at_the_row_position(kind, w):
    """Decoding the last S_q positions with ALiBi gives the prefill rows: the bias uses the row's
    position in the sequence, not its index among the new rows."""
    B, Hq, Hkv, S, d, S_q = 2, 4, 2, 17, 8, 3
    Qf, K, V = _rand((B, Hq, S, d), 16), _rand((B, Hkv, S, d), 17), _rand((B, Hkv, S, d), 18)
    slopes = [0.2, 0.4, 0.6, 0.8]
    O_ref, L_ref = oracle.attention(Qf, K, V, 0.3, kind, w, alibi=slopes)
    O, L = oracle.decode(Qf[:, :, S - S_q:], K, V, [S] * B, 0.3, kind, w, alibi=slopes)
    assert np.allclose(O, O_ref[:, :, S - S_q:], atol=1e-13, rtol=0)
    assert np.allclose(L, L_ref[:, :, S - S_q:], atol=1e-13, rtol=0)
