"""A given bias matrix b_ij added to the scores (attn_set_bias), GPU vs the fp64 oracle.

Every output is compared on small shapes: every mask kind (local + global with its global keys
and rows reading the bias at their own positions), the four broadcast shapes [Bb, Hb] of the
bias, ragged lengths with padded rows (the padding holds NaN, so a kernel that reads it into a
result fails), GQA and both head widths; the causal MHA 4K and the local + global 8K workloads
run at full size with a per-head bias, every output.  Bounds: those of the
bf16 forward (the bias is bf16, exact in the oracle's float32 copy, and adds one fp32
multiply-add per score).  The backward with the same bias is compared with the fp64 backward
oracle at the backward's bounds.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import all_rows, compare, gather_rows, small

pytestmark = pytest.mark.gpu

KINDS = (wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING)


def _bias(Bb, Hb, S, ld, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    b = (torch.randn(Bb, Hb, S, ld, generator=g) * scale).to(torch.bfloat16)
    b[..., S:] = float("nan")  # row padding: never part of a result
    return b


def _run(w, bias, Q, K, V):
    import transformer_self_attention_gb300 as tsa
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, scale=w.scale, kind=w.kind, window=w.window,
                         global_idx=list(w.globals_idx))
    plan.set_bias(bias.cuda())
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device=Q.device)
    plan(Q, K, V, O=O, LSE=LSE)
    torch.cuda.synchronize()
    st, code = plan.poll_device_error()
    assert st == 0 and code == 0, f"device error word {code}"
    return O, LSE, plan


def _check(w, Bb, Hb, ld, seed=3):
    Qc, Kc, Vc = wl.make_inputs(w)
    bias = _bias(Bb, Hb, w.S, ld, seed)
    O, LSE, _ = _run(w, bias, Qc.cuda(), Kc.cuda(), Vc.cuda())
    O_ref, L_ref = oracle.attention(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), w.scale, w.kind,
                                    w.window, list(w.globals_idx), bias=bias.float().numpy())
    return compare(w, O.float().cpu().numpy(), LSE.cpu().numpy(), O_ref, L_ref)


@pytest.mark.parametrize("Bb,Hb", [(1, 1), (2, 1), (1, 4), (2, 4)])
@pytest.mark.parametrize("kind", KINDS)
def test_bias_matrix_kinds_and_broadcasts(kind, Bb, Hb):
    _check(small("bm", 2, 4, 2, 300, 128, "bf16", kind, window=70), Bb, Hb, ld=304)


@pytest.mark.parametrize("S", [1, 8, 127, 128, 129, 257])
def test_bias_matrix_lengths(S):
    ld = (S + 7) // 8 * 8 + 8
    _check(small("bl", 1, 2, 2, S, 64, "bf16", wl.MASK_CAUSAL), 1, 2, ld=ld)


@pytest.mark.parametrize("d", [64, 128])
def test_bias_matrix_gqa(d):
    _check(small("bg", 2, 8, 2, 520, d, "bf16", wl.MASK_CAUSAL_SLIDING, window=129), 2, 8, ld=520)


def test_bias_matrix_minus_infinity_masks_keys():
    """A -inf bias above the diagonal on the full mask is the causal mask."""
    w = small("binf", 1, 2, 2, 200, 128, "bf16", wl.MASK_FULL)
    Qc, Kc, Vc = wl.make_inputs(w)
    tri = torch.zeros(1, 1, 200, 200)
    tri[0, 0] = torch.triu(torch.full((200, 200), float("-inf")), diagonal=1)
    O, LSE, _ = _run(w, tri.to(torch.bfloat16), Qc.cuda(), Kc.cuda(), Vc.cuda())
    O_ref, L_ref = oracle.attention(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), w.scale,
                                    wl.MASK_CAUSAL)
    compare(w, O.float().cpu().numpy(), LSE.cpu().numpy(), O_ref, L_ref)


def test_removing_the_bias_restores_the_plain_result():
    w = small("brm", 1, 2, 2, 300, 128, "bf16", wl.MASK_CAUSAL)
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    O1, L1, plan = _run(w, _bias(1, 1, 300, 304, 5), Q, K, V)
    plan.set_bias(None)
    O2, L2 = plan(Q, K, V)
    O_ref, L_ref = oracle.attention(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), w.scale, w.kind)
    torch.cuda.synchronize()
    compare(w, O2.float().cpu().numpy(), L2.cpu().numpy(), O_ref, L_ref)


@pytest.mark.parametrize("Bb,Hb", [(1, 1), (2, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_bias_matrix_local_global(d, Bb, Hb):
    """Local + global: the band tiles read the bias row by row, the gathered global keys one key at
    a time at their own positions, the global rows (their own items, key chunks merged) their own
    rows; globals at both ends and on both sides of tile edges."""
    _check(small("blg", 2, 4, 4, 520, d, "bf16", wl.MASK_LOCAL_GLOBAL, window=40,
                 globals_idx=(0, 127, 128, 300, 519)), Bb, Hb, ld=520)


@pytest.mark.parametrize("S", [1, 129, 300])
def test_bias_matrix_local_global_lengths(S):
    G = sorted({0, S // 2, S - 1})
    _check(small("blgl", 1, 2, 1, S, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=19, globals_idx=G), 1, 2,
           ld=(S + 7) // 8 * 8 + 8)


def test_bias_matrix_local_global_many_globals():
    """129 global tokens: two gathered key tiles per query tile and two global-row tiles."""
    _check(small("blgm", 1, 2, 2, 700, 128, "bf16", wl.MASK_LOCAL_GLOBAL, window=9,
                 globals_idx=list(range(3, 700, 5))[:129]), 1, 2, ld=704)


def test_bias_matrix_unsupported_and_invalid():
    import transformer_self_attention_gb300 as tsa
    bias = _bias(1, 1, 256, 256, 6).cuda()
    al = tsa.Attention(1, 2, 2, 256, 128, kind=wl.MASK_CAUSAL)
    al.set_alibi(wl.alibi_slopes(2))
    with pytest.raises(tsa.AttnError):
        al.set_bias(bias)
    pl = tsa.Attention(1, 2, 2, 256, 128, kind=wl.MASK_CAUSAL)
    with pytest.raises(tsa.AttnError):  # row stride not a multiple of 8
        pl.set_bias(_bias(1, 1, 256, 260, 7).cuda())
    with pytest.raises(tsa.AttnError):  # Hb neither 1 nor Hq
        pl.set_bias(_bias(1, 3, 256, 256, 7).cuda())
    pl.set_bias(bias)
    with pytest.raises(tsa.AttnError):  # ALiBi and a bias matrix together
        pl.set_alibi(wl.alibi_slopes(2))
    torch.cuda.synchronize()


# ------------------------------------------------------------------ backward with a bias matrix

def _check_backward(w, Bb, Hb, ld, seed=5):
    """dQ, dK, dV of the biased forward against the fp64 backward oracle with the same bias."""
    from test_gpu_backward import _cmp
    Qc, Kc, Vc = wl.make_inputs(w)
    dOc = wl.make_grad_output(w)
    bias = _bias(Bb, Hb, w.S, ld, seed)
    Q, K, V, dO = Qc.cuda(), Kc.cuda(), Vc.cuda(), dOc.cuda()
    O, LSE, plan = _run(w, bias, Q, K, V)
    dQ, dK, dV = (torch.full_like(t, float("nan")) for t in (Q, K, V))
    plan.backward(Q, K, V, O, LSE, dO, dQ, dK, dV)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    ref = oracle.backward(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), dOc.float().numpy(), w.scale,
                          w.kind, w.window, globals_idx=list(w.globals_idx), bias=bias.float().numpy())
    return [_cmp(n, g, r) for n, g, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref)]


@pytest.mark.parametrize("Bb,Hb", [(1, 1), (2, 1), (1, 4), (2, 4)])
@pytest.mark.parametrize("kind", KINDS)
def test_backward_bias_matrix_kinds_and_broadcasts(kind, Bb, Hb):
    """The bias enters the recomputed P of both backward kernels: the dQ kernel reads it along the
    query rows, the dK/dV kernel down the key columns; padded rows hold NaN."""
    _check_backward(small("bbm", 2, 4, 2, 300, 128, "bf16", kind, window=70), Bb, Hb, ld=304)


@pytest.mark.parametrize("S", [2, 129, 257])
def test_backward_bias_matrix_lengths_d64(S):
    ld = (S + 7) // 8 * 8 + 8
    _check_backward(small("bbl", 1, 2, 1, S, 64, "bf16", wl.MASK_CAUSAL), 1, 2, ld=ld)


def test_backward_bias_matrix_full_size_causal_mha_4k():
    """The causal MHA workload with a per-head bias [1, 32, S, S]: every gradient element against the
    oracle (one call per (batch, head) slice, exact for MHA)."""
    from test_gpu_backward import _cmp
    w = wl.CAUSAL_MHA_4K
    Qc, Kc, Vc = wl.make_inputs(w)
    dOc = wl.make_grad_output(w)
    g = torch.Generator().manual_seed(11)
    bias = (torch.randn(1, w.Hq, w.S, w.S, generator=g) * 2).to(torch.bfloat16)
    Q, K, V, dO = Qc.cuda(), Kc.cuda(), Vc.cuda(), dOc.cuda()
    O, LSE, plan = _run(w, bias, Q, K, V)
    dQ, dK, dV = (torch.full_like(t, float("nan")) for t in (Q, K, V))
    plan.backward(Q, K, V, O, LSE, dO, dQ, dK, dV)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    bf = bias.float().numpy()
    refs = [np.empty(t.shape, dtype=np.float64) for t in (dQ, dK, dV)]
    for b in range(w.B):
        for a in range(w.Hq):
            sl = lambda t: t[b:b + 1, a:a + 1].float().numpy()
            out = oracle.backward(sl(Qc), sl(Kc), sl(Vc), sl(dOc), w.scale, w.kind, bias=bf[:, a:a + 1])
            for r, x in zip(refs, out):
                r[b:b + 1, a:a + 1] = x
    for n, gr, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), refs):
        _cmp(f"{n} + bias matrix (every element)", gr, r)


def test_bias_matrix_full_size_causal_mha_4k():
    """The causal MHA workload (B 2, H 32, S 4096, d 128) with a per-head bias [1, 32, S, S] at
    full size: every output against the oracle."""
    w = wl.CAUSAL_MHA_4K
    Qc, Kc, Vc = wl.make_inputs(w)
    g = torch.Generator().manual_seed(11)
    bias = (torch.randn(1, w.Hq, w.S, w.S, generator=g) * 2).to(torch.bfloat16)
    O, LSE, _ = _run(w, bias, Qc.cuda(), Kc.cuda(), Vc.cuda())
    rows = all_rows(w)
    O_ref, L_ref = oracle.attention_rows(Kc.float().numpy(), Vc.float().numpy(), w.Hq, w.scale, w.kind, w.window,
                                         [], Qc.float().numpy().reshape(-1, w.d), rows[:, 0], rows[:, 1],
                                         rows[:, 2], bias=bias.float().numpy())
    compare(w, *gather_rows(O, LSE), O_ref, L_ref, report=f"{w.name} + bias matrix (every row)")


@pytest.mark.parametrize("Bb,Hb", [(1, 1), (2, 4)])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_bias_matrix_local_global(d, Bb, Hb):
    """Backward under local + global with a bias matrix: both kernels walk the partner lists and
    read b_ij along the row (dQ) or down the column (dK, dV) of every listed tile."""
    _check_backward(small("bblg", 2, 4, 2, 520, d, "bf16", wl.MASK_LOCAL_GLOBAL, window=40,
                          globals_idx=(0, 127, 128, 300, 519)), Bb, Hb, ld=520)


def test_bias_matrix_full_size_local_global_8k():
    """The 8K local + global workload (H 12, d 64, w 512, globals 0, 1000, 3000, 6000) with a per-head
    bias [1, 12, S, S] N(0, 2^2) at full size: every output against the oracle."""
    w = wl.LONGFORMER_8K
    Qc, Kc, Vc = wl.make_inputs(w)
    g = torch.Generator().manual_seed(12)
    bias = (torch.randn(1, w.Hq, w.S, w.S, generator=g) * 2).to(torch.bfloat16)
    O, LSE, _ = _run(w, bias, Qc.cuda(), Kc.cuda(), Vc.cuda())
    rows = all_rows(w)
    O_ref, L_ref = oracle.attention_rows(Kc.float().numpy(), Vc.float().numpy(), w.Hq, w.scale, w.kind, w.window,
                                         list(w.globals_idx), Qc.float().numpy().reshape(-1, w.d), rows[:, 0],
                                         rows[:, 1], rows[:, 2], bias=bias.float().numpy())
    compare(w, *gather_rows(O, LSE), O_ref, L_ref, report=f"{w.name} + bias matrix (every row)")
