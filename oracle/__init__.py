"""fp64 CPU oracle for masked scaled dot-product self-attention.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by bench.py's ``cpu_baseline`` leg and reference arm, never by the
library.  It shares no code with the CUDA path.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64); this module compiles
it with gcc on first use and marshals numpy arrays.  What it computes, per query
row i of head a (kv head g(a) = a // (Hq // Hkv)):

    s_ij = scale * q_i . k_j  over allowed j,   z_i = sum_j softmax_j(s_ij) v_j,
    LSE_i = ln sum_j exp(s_ij)

following "Trasformer 浅析" (atffang.github.io), sections 缩放点积注意力 and
填充掩码与因果掩码, and "Transformer 架构及其变体" (aaai.latere.ai), section
带显式形状的因果自注意力.

``decode`` is the key/value-cache form ("Trasformer 浅析", sections 推理：KV 缓存
and 交叉注意力; "第 8 章 现代大模型架构" (theaiera.top), section
预填充创建缓存，解码复用缓存): S_q new query rows per sequence at positions
cache_len[b] - S_q + i against the cache_len[b] cached keys and values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_FULL, MASK_CAUSAL, MASK_SLIDING, MASK_CAUSAL_SLIDING, MASK_LOCAL_GLOBAL = range(5)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so (gcc, OpenMP).  Returns the path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            lib.oracle_allowed.argtypes = [I, L, L, L, L, P]
            lib.oracle_allowed.restype = I
            lib.oracle_attention_rows.argtypes = [P, P, I, I, I, I, I, ctypes.c_double, I, I, P, I,
                                                  P, P, P, P, L, P, P]
            lib.oracle_attention_rows.restype = I
            lib.oracle_attention_rows_bias.argtypes = [P, P, I, I, I, I, I, ctypes.c_double, I, I, P, I, P,
                                                       P, P, P, P, L, P, P]
            lib.oracle_attention_rows_bias.restype = I
            lib.oracle_attention_rows_general.argtypes = [P, P, I, I, I, I, I, ctypes.c_double, I, I, P, I, P, P, I,
                                                          I, L, P, P, P, P, L, P, P]
            lib.oracle_attention_rows_general.restype = I
            lib.oracle_row_counts.argtypes = [I, I, I, P, I, P]
            lib.oracle_row_counts.restype = I
            lib.oracle_tile_classes.argtypes = [I, I, I, P, I, I, I, P]
            lib.oracle_tile_classes.restype = I
            lib.oracle_decode_allowed.argtypes = [I, L, L, L, L]
            lib.oracle_decode_allowed.restype = I
            lib.oracle_decode.argtypes = [P, P, P, I, I, I, I, I, I, ctypes.c_double, I, I, P, P, P]
            lib.oracle_decode.restype = I
            lib.oracle_decode_bias.argtypes = [P, P, P, I, I, I, I, I, I, ctypes.c_double, I, I, P, P, P, P]
            lib.oracle_decode_bias.restype = I
            lib.oracle_backward.argtypes = [P, P, P, P, I, I, I, I, I, ctypes.c_double, I, I, P, I, P, P, P, P]
            lib.oracle_backward.restype = I
            lib.oracle_backward_bias.argtypes = [P, P, P, P, I, I, I, I, I, ctypes.c_double, I, I, P, I, P, P, I, I, L,
                                                 P, P, P]
            lib.oracle_backward_bias.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _globals_array(globals_idx):
    g = np.ascontiguousarray(np.asarray(globals_idx if globals_idx is not None else [], dtype=np.int32))
    return g, int(g.size)


def _slopes(alibi, Hq):
    if alibi is None:
        return None
    a = np.ascontiguousarray(np.asarray(alibi, dtype=np.float64).reshape(-1))
    assert a.size == Hq
    return a


def attention_rows(K, V, Hq, scale, kind, window, globals_idx, Qrows, row_b, row_a, row_i, alibi=None,
                   bias=None):
    """Oracle outputs for an explicit list of rows.

    K, V: float32-castable arrays [B, Hkv, S, d]; Qrows: [n, d] query vectors of
    the rows; row_b / row_a / row_i: [n] batch, query head and position.
    alibi: optional [Hq] slopes m_a of the additive bias -m_a |i - j|.
    bias: optional float32-castable [Bb, Hb, S, ld] bias matrix added to the scaled
    scores (Bb in {1, B}, Hb in {1, Hq}: size 1 broadcasts; ld >= S).
    Returns (O [n, d] float64, LSE [n] float64).
    """
    lib = _load()
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    B, Hkv, S, d = K.shape
    Qrows = np.ascontiguousarray(Qrows, dtype=np.float32).reshape(-1, d)
    n = Qrows.shape[0]
    rb = np.ascontiguousarray(row_b, dtype=np.int32)
    ra = np.ascontiguousarray(row_a, dtype=np.int32)
    ri = np.ascontiguousarray(row_i, dtype=np.int32)
    assert rb.size == n and ra.size == n and ri.size == n
    g, ng = _globals_array(globals_idx)
    O = np.empty((n, d), dtype=np.float64)
    LSE = np.empty((n,), dtype=np.float64)
    sl = _slopes(alibi, Hq)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        Bb, Hb, Sb, ld = bias.shape
        assert Sb == S and Bb in (1, B) and Hb in (1, Hq) and ld >= S
    else:
        Bb = Hb = 1
        ld = 0
    rc = lib.oracle_attention_rows_general(_ptr(K), _ptr(V), B, Hq, Hkv, S, d, float(scale), int(kind),
                                           int(window), _ptr(g), ng, _ptr(sl) if sl is not None else None,
                                           _ptr(bias) if bias is not None else None, Bb, Hb, ld,
                                           _ptr(Qrows), _ptr(rb), _ptr(ra), _ptr(ri), n, _ptr(O), _ptr(LSE))
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return O, LSE


def attention(Q, K, V, scale, kind, window=0, globals_idx=None, alibi=None, bias=None):
    """Whole-tensor oracle: Q [B, Hq, S, d], K/V [B, Hkv, S, d] -> (O [B,Hq,S,d], LSE [B,Hq,S]) fp64."""
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    B, Hq, S, d = Q.shape
    bb, aa, ii = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(S), indexing="ij")
    O, LSE = attention_rows(K, V, Hq, scale, kind, window, globals_idx, Q.reshape(-1, d),
                            bb.ravel(), aa.ravel(), ii.ravel(), alibi=alibi, bias=bias)
    return O.reshape(B, Hq, S, d), LSE.reshape(B, Hq, S)


def allowed(kind, i, j, S, window, globals_idx=None) -> bool:
    """The oracle's mask predicate for one (i, j) pair."""
    lib = _load()
    flags = np.zeros(max(S, 1), dtype=np.uint8)
    if globals_idx is not None:
        for t in globals_idx:
            if 0 <= t < S:
                flags[t] = 1
    return bool(lib.oracle_allowed(int(kind), int(i), int(j), int(S), int(window), _ptr(flags)))


def row_counts(kind, S, window=0, globals_idx=None) -> np.ndarray:
    """Allowed keys per row, by enumeration of every (i, j)."""
    lib = _load()
    g, ng = _globals_array(globals_idx)
    out = np.empty((S,), dtype=np.int64)
    if lib.oracle_row_counts(int(kind), int(S), int(window), _ptr(g), ng, _ptr(out)) != 0:
        raise ValueError("oracle_row_counts failed")
    return out


def tile_classes(kind, S, window=0, globals_idx=None, tm=128, tn=128) -> np.ndarray:
    """Brute-force tile classes (0 SKIP, 1 FULL, 2 PARTIAL) over the S x S pair grid."""
    lib = _load()
    g, ng = _globals_array(globals_idx)
    out = np.empty(((S + tm - 1) // tm, (S + tn - 1) // tn), dtype=np.uint8)
    if lib.oracle_tile_classes(int(kind), int(S), int(window), _ptr(g), ng, int(tm), int(tn), _ptr(out)) != 0:
        raise ValueError("oracle_tile_classes failed")
    return out


def decode_allowed(kind, t, j, L, window=0) -> bool:
    """The decode mask predicate: query at position t, key j, cache length L."""
    return bool(_load().oracle_decode_allowed(int(kind), int(t), int(j), int(L), int(window)))


def decode(Q, K, V, cache_len, scale, kind, window=0, alibi=None):
    """Key/value-cache attention.

    Q [B, Hq, S_q, d]; K, V [B, Hkv, S_cap, d] (the cache); cache_len [B] ints.
    Row i of sequence b sits at position cache_len[b] - S_q + i.  Kinds FULL
    (cross-attention: every cached key), CAUSAL and CAUSAL_SLIDING.
    Returns (O [B, Hq, S_q, d], LSE [B, Hq, S_q]) in float64.
    """
    lib = _load()
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    B, Hq, S_q, d = Q.shape
    Bk, Hkv, S_cap, dk = K.shape
    assert Bk == B and dk == d and V.shape == K.shape
    lens = np.ascontiguousarray(np.asarray(cache_len, dtype=np.int32).reshape(-1))
    assert lens.size == B
    O = np.empty((B, Hq, S_q, d), dtype=np.float64)
    LSE = np.empty((B, Hq, S_q), dtype=np.float64)
    sl = _slopes(alibi, Hq)
    rc = lib.oracle_decode_bias(_ptr(Q), _ptr(K), _ptr(V), B, Hq, Hkv, S_q, S_cap, d, float(scale), int(kind),
                                int(window), _ptr(lens), _ptr(sl) if sl is not None else None, _ptr(O), _ptr(LSE))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return O, LSE


def backward(Q, K, V, dO, scale, kind, window=0, globals_idx=None, alibi=None, bias=None):
    """Gradients of the attention with respect to Q, K, V for the output gradient dO.

    Q, dO [B, Hq, S, d]; K, V [B, Hkv, S, d].  Returns (dQ, dK, dV) in float64 with the
    shapes of Q, K, V (dK and dV summed over the query heads of each kv head).
    bias: optional float32-castable [Bb, Hb, S, ld] bias matrix added to the scaled scores, as
    for attention_rows.
    """
    lib = _load()
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    dO = np.ascontiguousarray(dO, dtype=np.float32)
    B, Hq, S, d = Q.shape
    Hkv = K.shape[1]
    assert K.shape == V.shape == (B, Hkv, S, d) and dO.shape == Q.shape
    g, ng = _globals_array(globals_idx)
    sl = _slopes(alibi, Hq)
    dQ = np.empty(Q.shape, dtype=np.float64)
    dK = np.empty(K.shape, dtype=np.float64)
    dV = np.empty(V.shape, dtype=np.float64)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        Bb, Hb, Sb, ld = bias.shape
        assert Sb == S and Bb in (1, B) and Hb in (1, Hq) and ld >= S
    else:
        Bb = Hb = 1
        ld = 0
    rc = lib.oracle_backward_bias(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, Hq, Hkv, S, d, float(scale), int(kind),
                                  int(window), _ptr(g), ng, _ptr(sl) if sl is not None else None,
                                  _ptr(bias) if bias is not None else None, Bb, Hb, ld, _ptr(dQ), _ptr(dK),
                                  _ptr(dV))
    if rc != 0:
        raise ValueError("oracle_backward rejected its arguments")
    return dQ, dK, dV
