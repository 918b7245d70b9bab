"""The ALiBi score bias on the GPU (prefill and decode) vs the fp64 oracle with the same bias."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import all_rows, compare, gather_rows, small

pytestmark = pytest.mark.gpu

KINDS = (wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING)


def _run_prefill(w, slopes, Q, K, V):
    import transformer_self_attention_gb300 as tsa
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype=w.dtype, scale=w.scale, kind=w.kind, window=w.window)
    plan.set_alibi(slopes)
    O = torch.full_like(Q, float("nan"))
    L = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device=Q.device)
    plan(Q, K, V, O=O, LSE=L)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    return O, L, plan


def _full(w, slopes):
    Qc, Kc, Vc = wl.make_inputs(w)
    O, L, _ = _run_prefill(w, slopes, Qc.cuda(), Kc.cuda(), Vc.cuda())
    O_ref, L_ref = oracle.attention(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), w.scale, w.kind,
                                    w.window, alibi=slopes)
    return compare(w, O.float().cpu().numpy().reshape(-1, w.d), L.cpu().numpy().ravel(), O_ref.reshape(-1, w.d),
                   L_ref.ravel())


@pytest.mark.parametrize("S", [1, 129, 300])
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("d", [64, 128])
def test_prefill_alibi_kinds(kind, S, d):
    _full(small("a", 1, 4, 2, S, d, "bf16", kind, window=37), wl.alibi_slopes(4))


def test_prefill_alibi_steep_and_mixed_slopes():
    """Very different slopes per head, including zero and a steep one."""
    _full(small("m", 2, 4, 4, 400, 128, "bf16", wl.MASK_CAUSAL), [0.0, 0.01, 0.5, 4.0])


def test_prefill_alibi_fp32():
    _full(small("f", 1, 4, 4, 256, 64, "f32", wl.MASK_FULL), wl.alibi_slopes(4))


def test_prefill_alibi_removed_gives_the_unbiased_output():
    import transformer_self_attention_gb300 as tsa
    w = small("r", 1, 4, 2, 300, 128, "bf16", wl.MASK_CAUSAL)
    Q, K, V = (t.cuda() for t in wl.make_inputs(w))
    plain = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, kind=w.kind)
    O0, L0 = plain(Q, K, V)
    O1, L1, plan = _run_prefill(w, wl.alibi_slopes(4), Q, K, V)
    plan.set_alibi(None)
    O2, L2 = plan(Q, K, V)
    torch.cuda.synchronize()
    assert torch.equal(O0, O2) and torch.equal(L0, L2)
    assert not torch.equal(O0, O1)


def _full_lg(w, slopes):
    """Local + global with ALiBi: the global keys and rows take the distance term of their positions."""
    import transformer_self_attention_gb300 as tsa
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype=w.dtype, scale=w.scale, kind=w.kind, window=w.window,
                         global_idx=list(w.globals_idx))
    plan.set_alibi(slopes)
    O = torch.full_like(Q, float("nan"))
    L = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device=Q.device)
    plan(Q, K, V, O=O, LSE=L)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    O_ref, L_ref = oracle.attention(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), w.scale, w.kind,
                                    w.window, list(w.globals_idx), alibi=slopes)
    return compare(w, O.float().cpu().numpy().reshape(-1, w.d), L.cpu().numpy().ravel(), O_ref.reshape(-1, w.d),
                   L_ref.ravel())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [[0], [0, 300, 599], [5, 127, 128, 500], list(range(3, 600, 7))])
def test_prefill_alibi_local_global(G, d):
    """Gathered global keys (narrow tiles), chunked global rows and band tiles with the ALiBi term."""
    _full_lg(small("alg", 1, 4, 2, 600, d, "bf16", wl.MASK_LOCAL_GLOBAL, window=40, globals_idx=G),
             wl.alibi_slopes(4))


def test_prefill_alibi_local_global_steep_and_fp32():
    _full_lg(small("algs", 2, 3, 3, 520, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=33, globals_idx=(0, 260, 519)),
             [0.0, 0.05, 1.0])
    _full_lg(small("algf", 1, 2, 2, 300, 64, "f32", wl.MASK_LOCAL_GLOBAL, window=20, globals_idx=(0, 150)),
             [0.02, 0.3])


def test_prefill_alibi_local_global_full_size():
    """The local + global workload (H12 S8192 d64 w512, 4 globals) with geometric slopes; every output."""
    _full_lg(wl.LONGFORMER_8K, wl.alibi_slopes(wl.LONGFORMER_8K.Hq))


def test_prefill_alibi_full_size_causal_4k():
    """The 4K causal workload with geometric slopes, in the bench's launch configuration; every output."""
    w = wl.CAUSAL_MHA_4K
    slopes = wl.alibi_slopes(w.Hq)
    Qc, Kc, Vc = wl.make_inputs(w)
    O, L, _ = _run_prefill(w, slopes, Qc.cuda(), Kc.cuda(), Vc.cuda())
    rows = all_rows(w)
    O_ref, L_ref = oracle.attention_rows(Kc.float().numpy(), Vc.float().numpy(), w.Hq, w.scale, w.kind, w.window, None,
                                         Qc.float().numpy().reshape(-1, w.d), rows[:, 0], rows[:, 1], rows[:, 2],
                                         alibi=slopes)
    compare(w, *gather_rows(O, L), O_ref, L_ref, report=f"{w.name} + ALiBi (every row)")


# ------------------------------------------------------------------ decode

def _decode(w, slopes, grid_limit=None):
    import transformer_self_attention_gb300 as tsa
    Qc, Kc, Vc, lens = wl.make_decode_inputs(w, stale_fill=float("nan"))
    plan = tsa.DecodeAttention(w.B, w.Hq, w.Hkv, w.S_q, w.S_cap, w.d, scale=w.scale, kind=w.kind, window=w.window)
    plan.set_alibi(slopes)
    if grid_limit:
        plan.set_grid_limit(grid_limit)
    O = torch.full((w.B, w.Hq, w.S_q, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    L = torch.full((w.B, w.Hq, w.S_q), float("nan"), dtype=torch.float32, device="cuda")
    plan(Qc.cuda(), Kc.cuda(), Vc.cuda(), lens, O=O, LSE=L)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens, w.scale, w.kind,
                                 w.window, alibi=slopes)
    wb = small("x", 1, 1, 1, 1, w.d, "bf16", wl.MASK_FULL)  # tolerances of the bf16 path
    return compare(wb, O.float().cpu().numpy().reshape(-1, w.d), L.cpu().numpy().ravel(), O_ref.reshape(-1, w.d),
                   L_ref.ravel())


@pytest.mark.parametrize("limit", [None, 3])
@pytest.mark.parametrize("kind", [wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_CAUSAL_SLIDING])
def test_decode_alibi(kind, limit):
    w = wl.DecodeWorkload("da", 4, 8, 2, 2, 1500, 128, kind, window=600, seed=31, len_min=300)
    _decode(w, wl.alibi_slopes(8), grid_limit=limit)


@pytest.mark.parametrize("Hq,Hkv,S_q,d", [(32, 1, 1, 64), (8, 2, 8, 128)])
def test_decode_alibi_row_widths(Hq, Hkv, S_q, d):
    w = wl.DecodeWorkload("dr", 3, Hq, Hkv, S_q, 900, d, wl.MASK_CAUSAL, seed=32, len_min=S_q + 100)
    _decode(w, wl.alibi_slopes(Hq), grid_limit=5)


def test_decode_alibi_full_size_gqa_32k():
    _decode(wl.DECODE_GQA_32K, wl.alibi_slopes(wl.DECODE_GQA_32K.Hq))
