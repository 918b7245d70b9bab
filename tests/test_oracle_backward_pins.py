"""Pins of the fp64 backward oracle (gradients of the attention with respect to Q, K, V).

The pages state no backward formulas, only that the tiled method is exact and trains
models; the oracle is therefore the plain derivative of the forward definition.  It is
pinned here against float64 torch autograd through an independently written forward,
against central finite differences of the already-pinned forward oracle, and against
identities of the softmax.  No GPU.
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


def _torch_grads(Q, K, V, dO, scale, kind, w, G, slopes=None, bias=None):
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    M = torch.zeros(S, S, dtype=torch.bool)
    for i in range(S):
        for j in range(S):
            M[i, j] = oracle.allowed(kind, i, j, S, w, G)
    q = torch.from_numpy(Q).double().requires_grad_()
    k = torch.from_numpy(K).double().requires_grad_()
    v = torch.from_numpy(V).double().requires_grad_()
    kr = k.repeat_interleave(Hq // Hkv, dim=1)
    vr = v.repeat_interleave(Hq // Hkv, dim=1)
    s = q @ kr.transpose(-1, -2) * scale
    if slopes is not None:
        dist = (torch.arange(S)[:, None] - torch.arange(S)[None, :]).abs().double()
        s = s - torch.tensor(slopes, dtype=torch.float64)[None, :, None, None] * dist
    if bias is not None:  # [Bb, Hb, S, ld]: broadcast over batch / heads, padding columns unused
        s = s + torch.from_numpy(bias).double()[..., :S]
    s = s.masked_fill(~M, float("-inf"))
    o = torch.softmax(s, -1) @ vr
    (o * torch.from_numpy(dO).double()).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("Hkv", [1, 2, 4])
def test_backward_matches_autograd(kind, Hkv):
    B, Hq, S, d = 2, 4, 23, 6
    Q, K, V, dO = _rand((B, Hq, S, d), 1), _rand((B, Hkv, S, d), 2), _rand((B, Hkv, S, d), 3), _rand((B, Hq, S, d), 4)
    G = [0, 11] if kind == oracle.MASK_LOCAL_GLOBAL else None
    got = oracle.backward(Q, K, V, dO, 0.4, kind, 3, G)
    ref = _torch_grads(Q, K, V, dO, 0.4, kind, 3, G)
    for a, b in zip(got, ref):
        assert np.allclose(a, b, atol=1e-11, rtol=0)


@pytest.mark.parametrize("kind", [oracle.MASK_CAUSAL, oracle.MASK_SLIDING])
def test_backward_with_alibi_matches_autograd(kind):
    B, Hq, S, d = 1, 2, 19, 4
    Q, K, V, dO = _rand((B, Hq, S, d), 5), _rand((B, Hq, S, d), 6), _rand((B, Hq, S, d), 7), _rand((B, Hq, S, d), 8)
    got = oracle.backward(Q, K, V, dO, 0.5, kind, 4, alibi=[0.3, 1.1])
    ref = _torch_grads(Q, K, V, dO, 0.5, kind, 4, None, slopes=[0.3, 1.1])
    for a, b in zip(got, ref):
        assert np.allclose(a, b, atol=1e-11, rtol=0)


@pytest.mark.parametrize("kind", [oracle.MASK_CAUSAL, oracle.MASK_LOCAL_GLOBAL])
def test_backward_matches_finite_differences(kind):
    """Central differences of L = sum(O * dO) through the forward oracle (fp64 inputs widened from
    float32, so the perturbation h is applied to float64 copies through a scaled problem)."""
    B, Hq, Hkv, S, d = 1, 2, 1, 9, 3
    Q, K, V, dO = _rand((B, Hq, S, d), 9), _rand((B, Hkv, S, d), 10), _rand((B, Hkv, S, d), 11), _rand((B, Hq, S, d), 12)
    G = [4] if kind == oracle.MASK_LOCAL_GLOBAL else None
    dQ, dK, dV = oracle.backward(Q, K, V, dO, 0.7, kind, 2, G)

    def loss(Qx, Kx, Vx):
        O, _ = oracle.attention(Qx, Kx, Vx, 0.7, kind, 2, G)
        return float((O * dO.astype(np.float64)).sum())

    # float32 inputs: use a step that is exact in float32 and second-order accurate
    h = 2.0 ** -10
    rng = np.random.default_rng(0)
    for name, X, grad in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        for _ in range(6):
            idx = tuple(int(rng.integers(n)) for n in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (float(Xp[idx]) - float(Xm[idx]))
            assert abs(fd - grad[idx]) < 2e-5, (name, idx, fd, grad[idx])


def test_backward_identities():
    """Rows of P sum to one: the dV of a kv head sums to the dO of its query rows, and a value
    constant over positions has no influence on the weights (dQ = dK = 0)."""
    B, Hq, Hkv, S, d = 2, 4, 2, 17, 5
    Q, K, dO = _rand((B, Hq, S, d), 13), _rand((B, Hkv, S, d), 14), _rand((B, Hq, S, d), 15)
    V = _rand((B, Hkv, S, d), 16)
    for kind in KINDS:
        G = [2, 9] if kind == oracle.MASK_LOCAL_GLOBAL else None
        _, _, dV = oracle.backward(Q, K, V, dO, 0.5, kind, 3, G)
        for b in range(B):
            for g in range(Hkv):
                rows = dO[b, g * 2:(g + 1) * 2].astype(np.float64).sum(axis=(0, 1))
                assert np.allclose(dV[b, g].sum(axis=0), rows, atol=1e-11)
        Vc = np.broadcast_to(np.arange(d, dtype=np.float32), V.shape).copy()
        dQ, dK, _ = oracle.backward(Q, K, Vc, dO, 0.5, kind, 3, G)
        assert np.abs(dQ).max() < 1e-12 and np.abs(dK).max() < 1e-12


def test_backward_gqa_is_the_group_sum_of_mha():
    B, Hq, Hkv, S, d = 1, 6, 2, 15, 4
    Q, K, V, dO = _rand((B, Hq, S, d), 17), _rand((B, Hkv, S, d), 18), _rand((B, Hkv, S, d), 19), _rand((B, Hq, S, d), 20)
    dQ, dK, dV = oracle.backward(Q, K, V, dO, 0.5, oracle.MASK_CAUSAL)
    Kr, Vr = np.repeat(K, 3, axis=1), np.repeat(V, 3, axis=1)
    dQm, dKm, dVm = oracle.backward(Q, Kr, Vr, dO, 0.5, oracle.MASK_CAUSAL)
    assert np.allclose(dQ, dQm, atol=1e-13)
    assert np.allclose(dK, dKm.reshape(B, Hkv, 3, S, d).sum(axis=2), atol=1e-12)
    assert np.allclose(dV, dVm.reshape(B, Hkv, 3, S, d).sum(axis=2), atol=1e-12)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("bshape", [(1, 1), (2, 1), (1, 4), (2, 4)])
def test_backward_with_bias_matrix_matches_autograd(kind, bshape):
    """A given bias matrix b_ij [Bb, Hb, S, ld] (batch / head broadcast, padded rows) in the logits:
    the oracle's gradients equal float64 autograd through an independently written forward."""
    B, Hq, Hkv, S, d = 2, 4, 2, 21, 5
    Q, K, V, dO = _rand((B, Hq, S, d), 11), _rand((B, Hkv, S, d), 12), _rand((B, Hkv, S, d), 13), _rand((B, Hq, S, d), 14)
    bias = _rand((bshape[0], bshape[1], S, S + 3), 15, scale=2.0)
    G = [0, 9] if kind == oracle.MASK_LOCAL_GLOBAL else None
    got = oracle.backward(Q, K, V, dO, 0.35, kind, 4, G, bias=bias)
    ref = _torch_grads(Q, K, V, dO, 0.35, kind, 4, G, bias=bias)
    for a, b in zip(got, ref):
        assert np.allclose(a, b, atol=1e-11, rtol=0)


def test_backward_bias_padding_columns_are_not_read():
    """Values in the padding columns of the bias rows (ld > S) change nothing (up to the order in which
    the threads' dK / dV partial sums are added)."""
    B, Hq, S, d = 1, 2, 17, 4
    Q, K, V, dO = _rand((B, Hq, S, d), 21), _rand((B, Hq, S, d), 22), _rand((B, Hq, S, d), 23), _rand((B, Hq, S, d), 24)
    bias = _rand((1, Hq, S, S + 5), 25)
    a = oracle.backward(Q, K, V, dO, 0.5, oracle.MASK_CAUSAL, bias=bias)
    bias2 = bias.copy()
    bias2[..., S:] = 1e30
    b = oracle.backward(Q, K, V, dO, 0.5, oracle.MASK_CAUSAL, bias=bias2)
    for x, y in zip(a, b):
        assert np.allclose(x, y, atol=1e-13, rtol=0)
