"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test would fail on a plausible mistake in the oracle: a dropped scale, a
wrong sign or index in the mask predicate, a transposed operand, a wrong g(a)
or a missing normalisation.  None of these tests touches a GPU.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from conftest import read_golden

KINDS = (oracle.MASK_FULL, oracle.MASK_CAUSAL, oracle.MASK_SLIDING, oracle.MASK_CAUSAL_SLIDING,
         oracle.MASK_LOCAL_GLOBAL)


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def _vec(tokens):
    return np.array([float(t) for t in tokens], dtype=np.float32)


# ---------------------------------------------------------------- worked examples

def test_softmax_worked_example_weights():
    """One query, three keys, V = I_3: the output row is the weight vector."""
    g = read_golden("softmax_worked_example.txt")
    q = _vec(g["q"][0])
    K = np.stack([_vec(g["k1"][0]), _vec(g["k2"][0]), _vec(g["k3"][0])])
    V = np.eye(3, dtype=np.float32)
    scale = float(g["scale"][0][0])
    tol = float(g["tolerance"][0][0])
    O, LSE = oracle.attention(q[None, None, None, :], K[None, None], V[None, None], scale,
                              oracle.MASK_FULL)
    w = O[0, 0, 0]
    printed = sorted(float(x) for x in g["printed_weights_k1_k2_k3"][0])
    read = [float(x) for x in g["read_weights_k1_k2_k3"][0]]
    assert np.allclose(sorted(w), printed, atol=tol)          # the printed multiset
    assert abs(w[1] - printed[2]) < tol                       # k2 as printed
    assert np.allclose(w, read, atol=tol)                     # the read assignment
    dots = [float(x) for x in g["printed_dot_products"][0]]
    assert LSE[0, 0, 0] == pytest.approx(math.log(sum(math.exp(s) for s in dots)), abs=1e-12)


def test_softmax_ranking_example():
    g = read_golden("softmax_ranking_example.txt")
    q = _vec(g["q"][0])
    K = np.stack([_vec(g["k1"][0]), _vec(g["k2"][0]), _vec(g["k3"][0])])
    V = np.eye(3, dtype=np.float32)
    O, _ = oracle.attention(q[None, None, None, :], K[None, None], V[None, None], 1.0, oracle.MASK_FULL)
    w = O[0, 0, 0]
    order = ["k%d" % (int(t) + 1) for t in np.argsort(-w)]
    assert order == g["printed_softmax_ranking"][0]


def test_sliding_window_example():
    g = read_golden("longformer_neighbourhoods.txt")
    w = int(g["swa_window"][0][0])
    row, _, lo, _, hi = g["swa_row"][0]
    row, lo, hi = int(row), int(lo), int(hi)
    S = 16
    seen = [j for j in range(S) if oracle.allowed(oracle.MASK_SLIDING, row, j, S, w)]
    assert seen == list(range(lo, hi + 1))
    assert len(seen) == 2 * w + 1
    # interior rows see exactly 2w+1 keys, edge rows fewer
    counts = oracle.row_counts(oracle.MASK_SLIDING, S, w)
    assert all(counts[i] == 2 * w + 1 for i in range(w, S - w))
    assert counts[0] == w + 1 and counts[S - 1] == w + 1


def test_longformer_example_neighbourhoods():
    g = read_golden("longformer_neighbourhoods.txt")
    S = int(g["S"][0][0])
    w = int(g["window"][0][0])
    G = [int(x) for x in g["globals"][0]]
    r5000 = next(r for r in g["row"] if r[0] == "5000")
    lo, hi, nglob = int(r5000[2]), int(r5000[4]), int(r5000[6])
    seen = [j for j in range(S) if oracle.allowed(oracle.MASK_LOCAL_GLOBAL, 5000, j, S, w, G)]
    expect = sorted(set(range(lo, hi + 1)) | set(G))
    assert seen == expect
    assert len(seen) == (hi - lo + 1) + nglob == 1029
    r3000 = next(r for r in g["row"] if r[0] == "3000")
    assert r3000[1] == "all"
    counts = oracle.row_counts(oracle.MASK_LOCAL_GLOBAL, S, w, G)
    assert counts[3000] == S
    # every global column is seen by every row
    for gj in G:
        assert all(oracle.allowed(oracle.MASK_LOCAL_GLOBAL, i, gj, S, w, G) for i in range(0, S, 97))


def test_local_global_pair_count_closed_form():
    """Inclusion-exclusion count of the Longformer workload vs enumeration."""
    w = wl.LONGFORMER_8K
    S, win, G = w.S, w.window, sorted(w.globals_idx)
    # window pairs: S(2w+1) minus the two clipped triangles
    window_pairs = S * (2 * win + 1) - win * (win + 1)

    def wc(i):
        return min(i + win, S - 1) - max(i - win, 0) + 1
    rows_extra = sum(S - wc(i) for i in G)
    cols_extra = sum((S - wc(j)) - sum(1 for i in G if i != j and abs(i - j) > win) for j in G)
    closed = window_pairs + rows_extra + cols_extra
    counts = oracle.row_counts(w.kind, S, win, G)
    assert int(counts.sum()) == closed == 8192492


@pytest.mark.parametrize("w", [wl.TINY_FULL_F32, wl.CAUSAL_MHA_4K, wl.LONGFORMER_8K,
                               wl.SWA_GQA_16K.with_(S=5000)], ids=lambda w: w.name)
def test_pair_counts_match_enumeration(w):
    counts = oracle.row_counts(w.kind, w.S, w.window, list(w.globals_idx))
    assert int(counts.sum()) == wl.allowed_pairs_per_head(w)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("kind", KINDS)
def test_rows_sum_to_one(kind):
    """V all ones: every output entry is 1 (the weights of a row sum to 1)."""
    B, H, S, d = 1, 2, 37, 8
    Q, K = _rand((B, H, S, d), 1, 2.0), _rand((B, H, S, d), 2)
    V = np.ones((B, H, S, d), dtype=np.float32)
    O, _ = oracle.attention(Q, K, V, 0.3, kind, window=5, globals_idx=[0, 17, 30])
    assert np.allclose(O, 1.0, atol=1e-14)


@pytest.mark.parametrize("kind", KINDS)
def test_constant_values_give_constant_output(kind):
    B, H, S, d = 2, 2, 29, 6
    Q, K = _rand((B, H, S, d), 3), _rand((B, H, S, d), 4)
    c = _rand((B, H, 1, d), 5)
    V = np.broadcast_to(c, (B, H, S, d)).copy()
    O, _ = oracle.attention(Q, K, V, 0.5, kind, window=3, globals_idx=[4])
    assert np.allclose(O, np.broadcast_to(c, O.shape), atol=1e-12)


def test_causal_row_zero_is_v0():
    B, H, S, d = 1, 3, 16, 8
    Q, K, V = _rand((B, H, S, d), 6), _rand((B, H, S, d), 7), _rand((B, H, S, d), 8)
    O, LSE = oracle.attention(Q, K, V, 0.25, oracle.MASK_CAUSAL)
    assert np.array_equal(O[:, :, 0], V[:, :, 0].astype(np.float64))
    s00 = 0.25 * np.einsum("bhd,bhd->bh", Q[:, :, 0].astype(np.float64), K[:, :, 0].astype(np.float64))
    assert np.allclose(LSE[:, :, 0], s00, atol=1e-12)


@pytest.mark.parametrize("kind", [oracle.MASK_CAUSAL, oracle.MASK_CAUSAL_SLIDING])
def test_causal_future_perturbation(kind):
    """Changing K/V at positions j > i leaves row i bit-identical."""
    B, H, S, d = 1, 2, 24, 8
    Q, K, V = _rand((B, H, S, d), 9), _rand((B, H, S, d), 10), _rand((B, H, S, d), 11)
    O1, L1 = oracle.attention(Q, K, V, 0.35, kind, window=6)
    t = 13
    K2, V2 = K.copy(), V.copy()
    K2[:, :, t + 1:] = _rand(K2[:, :, t + 1:].shape, 12, 5.0)
    V2[:, :, t + 1:] = _rand(V2[:, :, t + 1:].shape, 13, 5.0)
    O2, L2 = oracle.attention(Q, K2, V2, 0.35, kind, window=6)
    assert np.array_equal(O1[:, :, : t + 1], O2[:, :, : t + 1])
    assert np.array_equal(L1[:, :, : t + 1], L2[:, :, : t + 1])
    assert not np.allclose(O1[:, :, t + 1:], O2[:, :, t + 1:])


def test_permutation_equivariance_full_mask():
    """Attention(PX) = P Attention(X) for the full mask; a joint permutation of K,V rows is invisible."""
    B, H, S, d = 1, 2, 21, 8
    Q, K, V = _rand((B, H, S, d), 14), _rand((B, H, S, d), 15), _rand((B, H, S, d), 16)
    O, L = oracle.attention(Q, K, V, 0.4, oracle.MASK_FULL)
    perm = np.random.default_rng(17).permutation(S)
    Op, Lp = oracle.attention(Q[:, :, perm], K[:, :, perm], V[:, :, perm], 0.4, oracle.MASK_FULL)
    assert np.allclose(Op, O[:, :, perm], atol=1e-12)
    assert np.allclose(Lp, L[:, :, perm], atol=1e-12)
    perm2 = np.random.default_rng(18).permutation(S)
    Ok, _ = oracle.attention(Q, K[:, :, perm2], V[:, :, perm2], 0.4, oracle.MASK_FULL)
    assert np.allclose(Ok, O, atol=1e-12)


@pytest.mark.parametrize("Hkv", [1, 2, 6])
def test_gqa_equals_mha_with_repeated_heads(Hkv):
    """GQA with contiguous groups == MHA whose K/V heads are repeated per group (Hkv=1 is MQA)."""
    B, Hq, S, d = 2, 6, 19, 8
    Q = _rand((B, Hq, S, d), 19)
    K, V = _rand((B, Hkv, S, d), 20), _rand((B, Hkv, S, d), 21)
    Og, Lg = oracle.attention(Q, K, V, 0.3, oracle.MASK_CAUSAL)
    rep = Hq // Hkv
    Km, Vm = np.repeat(K, rep, axis=1), np.repeat(V, rep, axis=1)
    Om, Lm = oracle.attention(Q, Km, Vm, 0.3, oracle.MASK_CAUSAL)
    assert np.array_equal(Og, Om) and np.array_equal(Lg, Lm)
    if 1 < Hkv < Hq:  # a different head map (interleaved) must give a different result
        Ki, Vi = np.tile(K, (1, rep, 1, 1)), np.tile(V, (1, rep, 1, 1))
        Oi, _ = oracle.attention(Q, Ki, Vi, 0.3, oracle.MASK_CAUSAL)
        assert not np.allclose(Oi, Og)


# ---------------------------------------------------------------- library special case

def _explicit_mask(kind, S, w, G):
    """Mask matrix written out pair by pair from the pages' definitions."""
    M = np.full((S, S), -np.inf)
    for i in range(S):
        for j in range(S):
            if kind == oracle.MASK_FULL:
                ok = True
            elif kind == oracle.MASK_CAUSAL:
                ok = j <= i
            elif kind == oracle.MASK_SLIDING:
                ok = abs(i - j) <= w
            elif kind == oracle.MASK_CAUSAL_SLIDING:
                ok = 0 <= i - j <= w
            else:
                ok = abs(i - j) <= w or i in G or j in G
            if ok:
                M[i, j] = 0.0
    return M


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("S,d", [(1, 1), (2, 3), (7, 3), (33, 1), (64, 64)])
def test_oracle_matches_float64_torch_softmax(kind, S, d):
    """On tiny S the oracle equals float64 torch.softmax(scale QK^T + M) V with M enumerated."""
    B, Hq, Hkv = 1, 4, 2
    w, G = 2, [0, S // 2]
    Q, K, V = _rand((B, Hq, S, d), 22), _rand((B, Hkv, S, d), 23), _rand((B, Hkv, S, d), 24)
    scale = 1.0 / math.sqrt(d)
    O, LSE = oracle.attention(Q, K, V, scale, kind, window=w, globals_idx=G)
    M = torch.tensor(_explicit_mask(kind, S, w, set(G)))
    for a in range(Hq):
        q = torch.tensor(Q[0, a], dtype=torch.float64)
        k = torch.tensor(K[0, a // (Hq // Hkv)], dtype=torch.float64)
        v = torch.tensor(V[0, a // (Hq // Hkv)], dtype=torch.float64)
        logits = scale * (q @ k.T) + M
        ref = torch.softmax(logits, dim=-1) @ v
        assert np.allclose(O[0, a], ref.numpy(), atol=1e-12, rtol=1e-12)
        assert np.allclose(LSE[0, a], torch.logsumexp(logits, dim=-1).numpy(), atol=1e-12)


def test_blocked_online_softmax_equals_oracle():
    """Tiling + the online max/sum recurrence reaches the plain result (exactness of the tiled method).

    The recurrence (m_new = max(m_old, m_block); l_new = l_old e^(m_old-m_new) + l_block e^(m_block-m_new))
    is the one in "Transformer 演进与变体", section Flash Attention (在线 Softmax), and
    "Trasformer 浅析", section 长序列的三条优化路线.
    """
    B, H, S, d, T = 1, 2, 45, 16, 8
    Q, K, V = _rand((B, H, S, d), 25, 2.0), _rand((B, H, S, d), 26), _rand((B, H, S, d), 27)
    scale = 0.25
    for kind in KINDS:
        O, L = oracle.attention(Q, K, V, scale, kind, window=7, globals_idx=[3, 40])
        Mfull = _explicit_mask(kind, S, 7, {3, 40})
        for h in range(H):
            q, k, v = (x[0, h].astype(np.float64) for x in (Q, K, V))
            for i in range(S):
                m, l, acc = -np.inf, 0.0, np.zeros(d)
                for j0 in range(0, S, T):
                    s = scale * (k[j0:j0 + T] @ q[i]) + Mfull[i, j0:j0 + T]
                    mb = s.max()
                    if mb == -np.inf:
                        continue
                    mn = max(m, mb)
                    p = np.exp(s - mn)
                    corr = math.exp(m - mn) if m != -np.inf else 0.0
                    l = l * corr + p.sum()
                    acc = acc * corr + p @ v[j0:j0 + T]
                    m = mn
                assert np.allclose(acc / l, O[0, h, i], atol=1e-12)
                assert abs(m + math.log(l) - L[0, h, i]) < 1e-12


def test_scale_statistics_of_generator():
    """var(scale q.k) is about 1 for iid N(0,1) inputs ("Trasformer 浅析", 缩放因子的必要性)."""
    w = wl.TINY_FULL_F32
    Q, K, _ = wl.make_inputs(w)
    s = (Q[0, 0].double() @ K[0, 0].double().T) * w.scale
    assert 0.85 < float(s.var()) < 1.15


# ---------------------------------------------------------------- tile classes

def test_tile_classes_small_by_hand():
    # causal, S=5, 2x2 tiles: tile (0,0) rows 0-1 cols 0-1 -> (0,1) not allowed -> PARTIAL
    c = oracle.tile_classes(oracle.MASK_CAUSAL, 5, tm=2, tn=2)
    assert c.tolist() == [[2, 0, 0], [1, 2, 0], [2, 2, 2]]
    c = oracle.tile_classes(oracle.MASK_FULL, 4, tm=2, tn=2)
    assert c.tolist() == [[1, 1], [1, 1]]
