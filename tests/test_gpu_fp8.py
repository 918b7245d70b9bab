"""E4M3 (FP8) inputs on the GPU vs the fp64 oracle over the dequantised values.

The oracle attends over q8 * dq, k8 * dk, v8 * dv exactly.  The kernel differs from it
at a few rounding points only: P is rounded to E4M3 before the second product (with
the running max of the lazy rescale as its reference, so P <= 2^8), the row sums use
the unrounded fp32 weights, and O is rounded to bf16 at the end; the products of E4M3
values are exact and their sums fp32.

Tolerance.  A CPU model of exactly those rounding points (`_e4m3_model`: the kernel's
per-tile running max with its 2^8 threshold, E4M3 round-to-nearest-even of fp32 P, fp32
row sums, bf16 rounding of O) is run on the same inputs, and its error against the
oracle sets the bounds.  Where the model and the kernel take the same rounding decisions
their outputs agree to fp32 summation order, so:
  * relative L2 against the oracle <= 1.25 x the model's + 1e-3;
  * max-abs against the oracle <= 1.5 x the model's + 4e-3 (the worst element can come
    from a weight whose rounding falls the other way on a midpoint);
  * relative L2 between the GPU and the model <= 0.25 x the model's own error + 1e-3: the
    kernel must follow the model much more closely than the model follows the oracle, so
    a real regression (a lost tile, a wrong scale, a stale P) cannot hide inside the E4M3
    rounding error.
The floors cover cases where E4M3 rounding is exact, such as a single key.  LSE comes
from the fp32 weights and keeps the bf16 path's 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import LSE_ABS, REPORT, small

pytestmark = pytest.mark.gpu

MAX_ABS_FACTOR, REL_L2_FACTOR, TRACK_FACTOR = 1.5, 1.25, 0.25
FLOOR_MAX_ABS, FLOOR_REL_L2 = 4e-3, 1e-3
LOG2E = 1.4426950408889634


def _allowed(kind, S, window, G=()):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    if kind == wl.MASK_LOCAL_GLOBAL:
        g = np.zeros(S, dtype=bool)
        g[list(G)] = True
        return (np.abs(i - j) <= window) | g[:, None] | g[None, :]
    if kind == wl.MASK_FULL:
        return np.ones((S, S), dtype=bool)
    if kind == wl.MASK_CAUSAL:
        return j <= i
    if kind == wl.MASK_SLIDING:
        return np.abs(i - j) <= window
    if kind == wl.MASK_CAUSAL_SLIDING:
        return (j <= i) & (i - j <= window)
    raise ValueError(kind)


def _e4m3_model(w, Q8, K8, V8, dq, dk, dv, bias=None):
    """O as the E4M3 kernel rounds it (see the module docstring), float64 [B, Hq, S, d].

    The scores are fp32 sums of exact E4M3 products, as on the tensor core; the weights are
    fp32 exponentials rounded to E4M3; O is accumulated in float64 and rounded to bf16.  An
    optional bias matrix [Bb, Hb, S, >= S] (float32 values of the bf16 tensor) joins the
    scores in log2 units, x = s sl2 + b log2 e, as the kernel's pass 1 forms it."""
    q = Q8.float().numpy()
    k = K8.float().numpy()
    v = V8.float().double().numpy()
    B, Hq, S, d = q.shape
    g = Hq // k.shape[1]
    T = 128
    nt = (S + T - 1) // T
    ok = _allowed(w.kind, S, w.window, w.globals_idx)
    sl2 = np.float32(w.scale * dq * dk * LOG2E)
    out = np.empty((B, Hq, S, d), dtype=np.float64)
    for b in range(B):
        for a in range(Hq):
            x = np.full((S, nt * T), -np.inf, dtype=np.float32)
            sc = (q[b, a] @ k[b, a // g].T) * sl2
            if bias is not None:
                bm = bias[0 if bias.shape[0] == 1 else b, 0 if bias.shape[1] == 1 else a, :, :S]
                sc = sc + bm.astype(np.float32) * np.float32(LOG2E)
            x[:, :S] = np.where(ok, sc, np.float32(-np.inf))
            tmax = x.reshape(S, nt, T).max(axis=2)
            ref = np.empty_like(tmax)
            m = np.full(S, -np.inf, dtype=np.float32)
            for t in range(nt):  # the lazy rescale: the reference moves only when the max grows by > 2^8
                grow = tmax[:, t] > m + 8.0
                m = np.where(grow, tmax[:, t], m)
                ref[:, t] = m
            fin = np.isfinite(ref)
            refc = np.where(fin, ref, np.float32(0.0))
            p32 = np.exp2(x[:, :S] - np.repeat(refc, T, axis=1)[:, :S])
            pr = torch.from_numpy(p32).to(torch.float8_e4m3fn).double().numpy()
            fac = np.repeat(np.where(fin, np.exp2(refc.astype(np.float64) - m[:, None]), 0.0), T, axis=1)[:, :S]
            num = (pr * fac) @ v[b, a // g]
            den = (p32.astype(np.float64) * fac).sum(axis=1)
            out[b, a] = num / den[:, None] * dv
    return torch.from_numpy(out).float().to(torch.bfloat16).double().numpy()


def _run(w, bias=None):
    import transformer_self_attention_gb300 as tsa
    Q8, K8, V8, (dq, dk, dv) = wl.make_fp8_inputs(w)
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype="e4m3", scale=w.scale, kind=w.kind, window=w.window,
                         global_idx=list(w.globals_idx))
    plan.set_fp8_descale(dq, dk, dv)
    if bias is not None:
        plan.set_bias(bias.cuda())
    O = torch.full((w.B, w.Hq, w.S, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    L = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device="cuda")
    plan(Q8.cuda(), K8.cuda(), V8.cuda(), O=O, LSE=L)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    return O.float().cpu().numpy(), L.cpu().numpy(), (Q8, K8, V8, dq, dk, dv)


def _norms(O, O_ref):
    d = np.asarray(O, dtype=np.float64) - O_ref
    return float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(O_ref))


def _check(O, L, O_ref, L_ref, O_model, report=None, track=True):
    """track=False: the rounding model walks the keys in plain tile order, which the kernel does not
    do for local + global (gathered global keys first, global rows in key chunks), so the two need
    not take the same rounding decisions; the bounds against the oracle still come from the model."""
    assert np.isfinite(O).all() and np.isfinite(L).all()
    max_abs, rel = _norms(O.reshape(O_ref.shape), O_ref)
    m_abs, m_rel = _norms(O_model.reshape(O_ref.shape), O_ref)
    g_abs, g_rel = _norms(O.reshape(O_ref.shape), O_model.reshape(O_ref.shape))
    lse = float(np.abs(L.reshape(L_ref.shape) - L_ref).max())
    bound_abs = MAX_ABS_FACTOR * m_abs + FLOOR_MAX_ABS
    bound_rel = REL_L2_FACTOR * m_rel + FLOOR_REL_L2
    bound_track = TRACK_FACTOR * m_rel + FLOOR_REL_L2
    line = (f"rows {O_ref.shape[0] if O_ref.ndim == 2 else O_ref.size // O_ref.shape[-1]}  max-abs {max_abs:.3e} "
            f"(bound {bound_abs:.3e})  rel-L2 {rel:.3e} (bound {bound_rel:.3e})  LSE {lse:.3e}  "
            f"GPU vs rounding model rel-L2 {g_rel:.3e} (bound {bound_track:.3e}), max-abs {g_abs:.3e}")
    print("fp8 errors:", line)
    if report:
        REPORT[report] = line
    assert max_abs <= bound_abs and rel <= bound_rel and lse <= LSE_ABS, line
    if track:
        assert g_rel <= bound_track, line


@pytest.mark.parametrize("d", [128, 64])  # d = 64: 64-byte rows in the 64-byte swizzle layout
@pytest.mark.parametrize("S", [1, 129, 300])
@pytest.mark.parametrize("kind", [wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING])
def test_fp8_kinds(kind, S, d):
    w = small("f8", 2, 4, 2, S, d, "bf16", kind, window=37)
    O, L, (Q8, K8, V8, dq, dk, dv) = _run(w)
    O_ref, L_ref = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                    w.kind, w.window)
    _check(O, L, O_ref * dv, L_ref, _e4m3_model(w, Q8, K8, V8, dq, dk, dv))


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("Bb,Hb", [(1, 1), (2, 4)])
@pytest.mark.parametrize("kind", [wl.MASK_CAUSAL, wl.MASK_SLIDING])
def test_fp8_bias_matrix(kind, Bb, Hb, d):
    """E4M3 inputs with a bias matrix b_ij (bf16 N(0, 2^2), NaN row padding): the bias joins the
    descaled scores; bounds from the rounding model with the same bias."""
    w = small("f8b", 2, 4, 2, 300, d, "bf16", kind, window=37)
    g = torch.Generator().manual_seed(21)
    bias = (torch.randn(Bb, Hb, w.S, 304, generator=g) * 2).to(torch.bfloat16)
    bias[..., w.S:] = float("nan")
    O, L, (Q8, K8, V8, dq, dk, dv) = _run(w, bias)
    bf = bias.float().numpy()
    O_ref, L_ref = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                    w.kind, w.window, bias=bf)
    _check(O, L, O_ref * dv, L_ref, _e4m3_model(w, Q8, K8, V8, dq, dk, dv, bias=bf))


@pytest.mark.parametrize("d", [128, 64])  # d = 64: gathered rows written in the 64-byte swizzle layout
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("S,G", [(300, (0, 150, 299)), (700, tuple(range(3, 700, 5))[:129])])
def test_fp8_local_global(S, G, bias, d):
    """E4M3 under local + global: gathered global keys in E4M3 narrow tiles, global rows in key chunks;
    with and without a bias matrix."""
    w = small("f8lg", 1, 4, 2, S, d, "bf16", wl.MASK_LOCAL_GLOBAL, window=40, globals_idx=G)
    bm = None
    if bias:
        g = torch.Generator().manual_seed(22)
        bm = (torch.randn(1, 4, S, (S + 7) // 8 * 8, generator=g) * 2).to(torch.bfloat16)
        bm[..., S:] = float("nan")
    O, L, (Q8, K8, V8, dq, dk, dv) = _run(w, bm)
    bf = None if bm is None else bm.float().numpy()
    O_ref, L_ref = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                    w.kind, w.window, list(G), bias=bf)
    _check(O, L, O_ref * dv, L_ref, _e4m3_model(w, Q8, K8, V8, dq, dk, dv, bias=bf), track=False)


def _alibi_bias(slopes, S):
    """The ALiBi bias -m_a |i - j| as a [1, Hq, S, S] float32 matrix (the model's bias form)."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    return np.stack([-np.float32(m) * np.abs(i - j).astype(np.float32) for m in slopes])[None]


@pytest.mark.parametrize("kind,G,d", [(wl.MASK_CAUSAL, (), 128), (wl.MASK_SLIDING, (), 128),
                                      (wl.MASK_CAUSAL_SLIDING, (), 128), (wl.MASK_LOCAL_GLOBAL, (0, 150, 299), 128),
                                      (wl.MASK_CAUSAL, (), 64), (wl.MASK_SLIDING, (), 64),
                                      (wl.MASK_LOCAL_GLOBAL, (0, 150, 299), 64)])
def test_fp8_alibi(kind, G, d):
    """E4M3 inputs with ALiBi slopes: the distance term joins the descaled scores element by element;
    bounds from the rounding model given the same bias as a matrix."""
    import transformer_self_attention_gb300 as tsa
    w = small("f8a", 1, 4, 2, 300, d, "bf16", kind, window=37, globals_idx=G)
    slopes = wl.alibi_slopes(4)
    Q8, K8, V8, (dq, dk, dv) = wl.make_fp8_inputs(w)
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype="e4m3", scale=w.scale, kind=w.kind, window=w.window,
                         global_idx=list(G))
    plan.set_fp8_descale(dq, dk, dv)
    plan.set_alibi(slopes)
    O = torch.full((w.B, w.Hq, w.S, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    L = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device="cuda")
    plan(Q8.cuda(), K8.cuda(), V8.cuda(), O=O, LSE=L)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    O_ref, L_ref = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                    w.kind, w.window, list(G), alibi=slopes)
    model = _e4m3_model(w, Q8, K8, V8, dq, dk, dv, bias=_alibi_bias(slopes, w.S))
    _check(O.float().cpu().numpy(), L.cpu().numpy(), O_ref * dv, L_ref, model, track=kind != wl.MASK_LOCAL_GLOBAL)


def test_fp8_rounding_model_is_not_trivial():
    """The model's own error is the E4M3 rounding of P: well above bf16 rounding, well below
    the raw 2^-4 worst case, on the 300-token causal case."""
    w = small("f8m", 1, 2, 2, 300, 128, "bf16", wl.MASK_CAUSAL)
    Q8, K8, V8, (dq, dk, dv) = wl.make_fp8_inputs(w)
    O_ref, _ = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                w.kind, w.window)
    m_abs, m_rel = _norms(_e4m3_model(w, Q8, K8, V8, dq, dk, dv), O_ref * dv)
    assert 1e-3 < m_rel < 2.0 ** -4, m_rel


def test_fp8_full_size_causal_4k():
    """Every output of the causal 4K workload against the oracle, bounds from the model."""
    w = wl.CAUSAL_MHA_4K
    O, L, (Q8, K8, V8, dq, dk, dv) = _run(w)
    O_ref, L_ref = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                    w.kind, w.window)
    _check(O, L, O_ref * dv, L_ref, _e4m3_model(w, Q8, K8, V8, dq, dk, dv),
           report=f"{w.name} E4M3 (every row)")


def test_fp8_unsupported_combinations():
    import transformer_self_attention_gb300 as tsa
    plan = tsa.Attention(1, 2, 2, 256, 128, dtype="e4m3", kind=wl.MASK_CAUSAL)
    plan.set_alibi([0.1, 0.2])
    with pytest.raises(tsa.AttnError):  # ALiBi and a bias matrix are exclusive
        plan.set_bias(torch.zeros(1, 1, 256, 256, dtype=torch.bfloat16, device="cuda"))


def test_fp8_full_size_local_global_8k():
    """The 8K local + global workload (d 64) in E4M3: every output against the oracle, bounds from the
    rounding model (plain tile order: no tracking bound)."""
    w = wl.LONGFORMER_8K
    O, L, (Q8, K8, V8, dq, dk, dv) = _run(w)
    O_ref, L_ref = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                    w.kind, w.window, list(w.globals_idx))
    _check(O, L, O_ref * dv, L_ref, _e4m3_model(w, Q8, K8, V8, dq, dk, dv), report=f"{w.name} E4M3 (every row)",
           track=False)
