"""A given bias matrix b_ij added to the scores (attn_set_bias), GPU vs the fp64 oracle.

Every output is compared on small shapes: the four interval kinds, the four broadcast
shapes [Bb, Hb] of the bias, ragged lengths with padded rows (the padding holds NaN, so a
kernel that reads it into a result fails), GQA and both head widths; the causal MHA 4K
workload runs at full size with a per-head bias on sampled rows.  Bounds: those of the
bf16 forward (the bias is bf16, exact in the oracle's float32 copy, and adds one fp32
multiply-add per score).
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
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, scale=w.scale, kind=w.kind, window=w.window)
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
                                    w.window, bias=bias.float().numpy())
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


def test_bias_matrix_unsupported_and_invalid():
    import transformer_self_attention_gb300 as tsa
    bias = _bias(1, 1, 256, 256, 6).cuda()
    lg = tsa.Attention(1, 2, 2, 256, 128, kind=wl.MASK_LOCAL_GLOBAL, window=8, global_idx=[0])
    with pytest.raises(tsa.AttnError):
        lg.set_bias(bias)
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
    Q, K, V = (t.cuda() for t in wl.make_inputs(small("u", 1, 2, 2, 256, 128, "bf16", wl.MASK_CAUSAL)))
    O, LSE = pl(Q, K, V)
    with pytest.raises(tsa.AttnError):  # no backward with a bias matrix
        pl.backward(Q, K, V, O, LSE, O)
    torch.cuda.synchronize()


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
