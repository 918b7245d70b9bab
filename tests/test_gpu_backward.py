"""Backward pass on the GPU vs the fp64 backward oracle (dQ, dK, dV).

The forward runs first on the CUDA path (its O and LSE feed the backward, as in
training); the expected gradients are the oracle's, computed from Q, K, V and dO
alone.  Outputs are NaN-poisoned before each call, so an unwritten row fails.

Tolerance.  The kernels round O (the forward's output), P and dS to bf16 before the
products and round the gradients to bf16 at the end; everything else is fp32.  A CPU
model of exactly those rounding points against the fp64 gradients gives a normwise
relative error of 2.3e-3 to 2.5e-3 and a largest element error of 2.8e-3 to 4.5e-3 of
the largest |gradient| (S = 256 to 1024, d = 64 and 128, full and causal).  The bounds
are four times that: relative L2 <= 1e-2 and max |error| <= 2e-2 * max |gradient|.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import REPORT, small

pytestmark = pytest.mark.gpu

GRAD_REL_L2 = 1e-2
GRAD_MAX_REL = 2e-2
KINDS = (wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING)


def _plan(w):
    import transformer_self_attention_gb300 as tsa
    return tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype=w.dtype, scale=w.scale, kind=w.kind, window=w.window,
                         global_idx=list(w.globals_idx))


def _run(w, Q, K, V, dO, plan=None, alibi=None):
    plan = plan or _plan(w)
    if alibi is not None:
        plan.set_alibi(alibi)
    O, LSE = plan(Q, K, V)
    dQ, dK, dV = (torch.full_like(t, float("nan")) for t in (Q, K, V))
    plan.backward(Q, K, V, O, LSE, dO, dQ, dK, dV)
    torch.cuda.synchronize()
    st, code = plan.poll_device_error()
    assert st == 0 and code == 0, f"device error word {code}"
    return dQ, dK, dV, plan


def _cmp(name, got, ref, workload=wl.CAUSAL_MHA_4K.name):
    got = got.float().cpu().numpy().astype(np.float64) if torch.is_tensor(got) else got
    assert np.isfinite(got).all(), f"{name}: non-finite (unwritten?) gradient"
    diff = got - ref
    scale = max(float(np.abs(ref).max()), 1e-30)
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    mx = float(np.abs(diff).max()) / scale
    assert rel <= GRAD_REL_L2, f"{name}: relative L2 error {rel:.3e}"
    assert mx <= GRAD_MAX_REL, f"{name}: max error {mx:.3e} of max |ref|"
    print(f"GRADERR {name} rel_l2 {rel:.3e} max_rel {mx:.3e}")
    if "every element" in name:
        REPORT[f"{workload} backward {name}"] = (
            f"elements {ref.size}  max |error| / max |gradient| {mx:.3e}  rel-L2 {rel:.3e}")
    return rel, mx


def _check(w, alibi=None):
    Qc, Kc, Vc = wl.make_inputs(w)
    dOc = wl.make_grad_output(w)
    dQ, dK, dV, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), dOc.cuda(), alibi=alibi)
    ref = oracle.backward(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), dOc.float().numpy(), w.scale,
                          w.kind, w.window, globals_idx=list(w.globals_idx), alibi=alibi)
    one_key = w.S == 1 or (w.window == 0 and w.kind in (wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING))
    if one_key:
        # every row sees one key (S = 1, or a window of 0): the softmax is the constant 1, so the
        # exact dQ and dK are zero and dV_j = the group's dO_j; the kernel's dQ and dK
        # are the rounding of O to bf16 (D_i = dO_i . O_i against dO_i . v_i), far below 1e-4
        assert np.abs(ref[0]).max() == 0 and np.abs(ref[1]).max() == 0
        for g in (dQ, dK):
            assert torch.isfinite(g).all() and g.float().abs().max().item() <= 1e-4
        return [_cmp("dV", dV, ref[2])]
    return [_cmp(n, g, r) for n, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref)]


@pytest.mark.parametrize("S", [1, 127, 128, 129, 300])
@pytest.mark.parametrize("kind", KINDS)
def test_backward_kinds_and_ragged_lengths(kind, S):
    _check(small("b", 1, 2, 2, S, 128, "bf16", kind, window=37))


@pytest.mark.parametrize("Hkv", [1, 2, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_gqa_and_mqa(Hkv, d):
    """dK and dV of a kv head sum over the query heads of its group."""
    _check(small("g", 2, 8, Hkv, 257, d, "bf16", wl.MASK_CAUSAL))


@pytest.mark.parametrize("w_", [0, 1, 127, 128, 129, 255])
@pytest.mark.parametrize("kind", [wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING])
def test_backward_windows_straddling_tile_edges(kind, w_):
    _check(small("w", 1, 2, 1, 520, 64, "bf16", kind, window=w_))


def test_backward_many_query_tiles_per_key_tile():
    """Full mask over 1000 positions with 4 query heads per kv head: every key tile walks
    32 (head, query tile) pairs, with both pipeline stages reused many times."""
    _check(small("long", 1, 4, 1, 1000, 128, "bf16", wl.MASK_FULL))


def test_backward_repeated_calls_are_identical():
    """No atomics: the same bits every call."""
    w = small("rep", 2, 4, 2, 700, 128, "bf16", wl.MASK_CAUSAL)
    Q, K, V = (t.cuda() for t in wl.make_inputs(w))
    dO = wl.make_grad_output(w, "cuda")
    a = _run(w, Q, K, V, dO)
    b = _run(w, Q, K, V, dO, plan=a[3])
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


def test_backward_unsupported_configurations():
    """The backward takes bf16 plans only: an fp32 plan is refused before any launch."""
    import transformer_self_attention_gb300 as tsa
    w = small("u", 1, 2, 2, 256, 64, "f32", wl.MASK_CAUSAL)
    Q, K, V = (t.cuda() for t in wl.make_inputs(w))
    plan = tsa.Attention(1, 2, 2, 256, 64, dtype="f32", kind=wl.MASK_CAUSAL)
    O, LSE = plan(Q, K, V)
    with pytest.raises(tsa.AttnError) as e:
        plan.backward(Q, K, V, O, LSE, O)
    assert e.value.status == tsa.ATTN_ERR_UNSUPPORTED
    torch.cuda.synchronize()


# ------------------------------------------------------------------ local + global
# The window |i - j| <= w plus global tokens that attend to and are attended by every position
# ("Transformer 演进与变体", section 稀疏注意力).  Both kernels walk per-tile lists with a bit mask;
# a global row's dQ and a global key's dK, dV sum over every position.

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S,w_,G", [(1, 0, (0,)), (129, 5, (0, 128)), (300, 40, (0, 100, 299)),
                                    (520, 130, (0, 127, 128, 255, 519)), (700, 64, ())])
def test_backward_local_global(S, w_, G, d):
    """Global tokens at the ends and on both sides of tile edges, windows inside and across tiles,
    no global at all (the plain symmetric window through the list path)."""
    _check(small("blg", 1, 2, 2, S, d, "bf16", wl.MASK_LOCAL_GLOBAL, window=w_, globals_idx=G))


def test_backward_local_global_many_globals_gqa():
    """129 global tokens (more than a tile of them: every tile holds some, so every list is every
    tile) and a GQA group of 4: dK and dV of a kv head sum over the group."""
    _check(small("blgm", 2, 8, 2, 640, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=20,
                 globals_idx=tuple(range(0, 640, 5))[:129]))


def test_backward_local_global_whole_global_tile():
    """A whole 128-position tile of global tokens: every pair against it is allowed, so the list
    entries of the tiles outside its band are FULL (no mask) in both kernels."""
    _check(small("blgt", 1, 2, 1, 520, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=10,
                 globals_idx=tuple(range(128, 256))))


def test_backward_local_global_alibi():
    """ALiBi under local + global: -m_a |i - j| for the window and the global pairs alike."""
    _check(small("blga", 1, 4, 2, 600, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=40, globals_idx=(0, 333, 599)),
           alibi=wl.alibi_slopes(4))


def test_backward_local_global_full_size():
    """The 8K local + global workload (H 12, d 64, w 512, globals 0, 1000, 3000, 6000) at full size:
    every element of dQ, dK and dV against the oracle, one oracle call per head (exact for MHA),
    norms over the whole tensors."""
    w = wl.LONGFORMER_8K
    assert w.Hq == w.Hkv
    Qc, Kc, Vc = wl.make_inputs(w)
    dOc = wl.make_grad_output(w)
    dQ, dK, dV, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), dOc.cuda())
    refs = [np.empty(t.shape, dtype=np.float64) for t in (dQ, dK, dV)]
    for b in range(w.B):
        for a in range(w.Hq):
            sl = lambda t: t[b:b + 1, a:a + 1].float().numpy()
            out = oracle.backward(sl(Qc), sl(Kc), sl(Vc), sl(dOc), w.scale, w.kind, w.window,
                                  globals_idx=list(w.globals_idx))
            for r, x in zip(refs, out):
                r[b:b + 1, a:a + 1] = x
    for n, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), refs):
        _cmp(f"{n} (every element)", g, r, workload=w.name)


@pytest.mark.parametrize("S", [1, 129, 300])
@pytest.mark.parametrize("kind", KINDS)
def test_backward_alibi_kinds(kind, S):
    """ALiBi -m_a |i - j| in the forward: the backward recomputes P with it (symmetric kinds take
    the absolute value, the causal kinds see j <= i only); every gradient against the oracle."""
    _check(small("ba", 1, 4, 2, S, 128, "bf16", kind, window=37), alibi=wl.alibi_slopes(4))


@pytest.mark.parametrize("d", [64, 128])
def test_backward_alibi_gqa_steep_slopes(d):
    """Steep slopes (m_a up to 1): the bias dominates the scores and P is concentrated near the
    diagonal; GQA sums dK and dV over the group."""
    w = small("bas", 2, 8, 2, 400, d, "bf16", wl.MASK_CAUSAL)
    _check(w, alibi=[2.0 ** (-a / 2.0) for a in range(8)])


def test_backward_alibi_full_size_causal_mha_4k():
    """The 4K causal workload with geometric ALiBi slopes: every gradient element against the
    oracle (one call per (batch, head) slice, exact for MHA)."""
    w = wl.CAUSAL_MHA_4K
    slopes = wl.alibi_slopes(w.Hq)
    Qc, Kc, Vc = wl.make_inputs(w)
    dOc = wl.make_grad_output(w)
    dQ, dK, dV, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), dOc.cuda(), alibi=slopes)
    refs = [np.empty(t.shape, dtype=np.float64) for t in (dQ, dK, dV)]
    for b in range(w.B):
        for a in range(w.Hq):
            sl = lambda t: t[b:b + 1, a:a + 1].float().numpy()
            out = oracle.backward(sl(Qc), sl(Kc), sl(Vc), sl(dOc), w.scale, w.kind, alibi=[slopes[a]])
            for r, x in zip(refs, out):
                r[b:b + 1, a:a + 1] = x
    for n, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), refs):
        _cmp(f"{n} + ALiBi (every element)", g, r)


def test_backward_full_size_causal_mha_4k():
    """The causal MHA workload (B 2, H 32, S 4096, d 128) at full size, in the launch
    configuration bench.py times: every element of dQ, dK and dV against the oracle (one
    oracle call per (batch, head) slice, exact for MHA), with the norms taken over the whole
    tensors; and the identities that hold at any size -- the rows of P sum to one, so
    sum_j dV_j = sum_i dO_i, and the rows of dS sum to zero, so sum_j dK_j = 0."""
    w = wl.CAUSAL_MHA_4K
    assert w.Hq == w.Hkv
    Qc, Kc, Vc = wl.make_inputs(w)
    dOc = wl.make_grad_output(w)
    dQ, dK, dV, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), dOc.cuda())
    for t in (dQ, dK, dV):
        assert torch.isfinite(t).all()
    refs = [np.empty(t.shape, dtype=np.float64) for t in (dQ, dK, dV)]
    for b in range(w.B):
        for a in range(w.Hq):
            sl = lambda t: t[b:b + 1, a:a + 1].float().numpy()
            for r, x in zip(refs, oracle.backward(sl(Qc), sl(Kc), sl(Vc), sl(dOc), w.scale, w.kind)):
                r[b:b + 1, a:a + 1] = x
    for n, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), refs):
        _cmp(f"{n} (every element)", g, r)
    # identities on every head (fp64 sums of the bf16 gradients)
    dV64 = dV.double().sum(dim=2)
    dO64 = dOc.double().cuda().sum(dim=2)
    err = (dV64 - dO64).abs().max().item()
    assert err <= GRAD_MAX_REL * dO64.abs().max().item(), f"sum_j dV_j vs sum_i dO_i: {err:.3e}"
    dK64 = dK.double()
    resid = dK64.sum(dim=2).abs().max().item()
    assert resid <= GRAD_MAX_REL * dK64.abs().sum(dim=2).max().item(), f"sum_j dK_j: {resid:.3e}"
