"""Decode / key-value-cache attention on the GPU vs the fp64 decode oracle (every output).

The stale part of every cache (positions at or past a sequence's length) is filled
with NaN, so a kernel that reads a stale key or value fails the finiteness check.
Outputs are NaN-poisoned before each call, so an unwritten row fails too.  Small
shapes cover every kind, both head widths, the 16/32/64 packed-row widths, ragged
lengths on and off tile edges, one-position caches and sequences split into many
key chunks (merged on the device); the five decode workloads run at full size in
the launch configuration bench.py times.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import BF16_MAX_ABS, BF16_REL_L2, LSE_ABS

pytestmark = pytest.mark.gpu


def _run(w, Q, K, V, lens, plan=None, reps=1, grid_limit=None):
    import transformer_self_attention_gb300 as tsa
    if plan is None:
        plan = tsa.DecodeAttention(w.B, w.Hq, w.Hkv, w.S_q, w.S_cap, w.d, scale=w.scale, kind=w.kind,
                                   window=w.window)
    if grid_limit:
        plan.set_grid_limit(grid_limit)
    out = []
    for _ in range(reps):
        O = torch.full_like(Q, float("nan"))
        LSE = torch.full((w.B, w.Hq, w.S_q), float("nan"), dtype=torch.float32, device=Q.device)
        plan(Q, K, V, lens, O=O, LSE=LSE)
        torch.cuda.synchronize()
        st, code = plan.poll_device_error()
        assert st == 0 and code == 0, f"device error word {code}"
        out.append((O.float().cpu().numpy(), LSE.cpu().numpy()))
    return out, plan


def _compare(O, LSE, O_ref, L_ref):
    assert np.isfinite(O).all(), "non-finite output (stale cache read or unwritten row)"
    assert np.isfinite(LSE).all(), "non-finite LSE"
    diff = O.astype(np.float64) - O_ref
    max_abs = float(np.abs(diff).max())
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(O_ref), 1e-30))
    lse = float(np.abs(LSE.astype(np.float64) - L_ref).max())
    assert max_abs <= BF16_MAX_ABS, f"max abs error {max_abs:.3e}"
    assert rel <= BF16_REL_L2, f"relative L2 error {rel:.3e}"
    assert lse <= LSE_ABS, f"LSE error {lse:.3e}"
    return max_abs, rel, lse


def _check(w, reps=1, grid_limit=None):
    Qc, Kc, Vc, lens = wl.make_decode_inputs(w, stale_fill=float("nan"))
    outs, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), lens, reps=reps, grid_limit=grid_limit)
    O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens, w.scale,
                                 w.kind, w.window)
    res = [_compare(O, LSE, O_ref, L_ref) for O, LSE in outs]
    if reps > 1:  # the same bits every call (the arrival counters wrap back to zero)
        assert all(np.array_equal(outs[0][0], o) and np.array_equal(outs[0][1], l) for o, l in outs[1:])
    return res[0]


def _dw(name, B, Hq, Hkv, S_q, S_cap, d, kind, window=0, len_min=0, seed=21):
    return wl.DecodeWorkload(name, B, Hq, Hkv, S_q, S_cap, d, kind, window=window, seed=seed, len_min=len_min)


@pytest.mark.parametrize("kind", [wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_CAUSAL_SLIDING])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_kinds_ragged(kind, d):
    """Ragged lengths in [S_q, 700]: chunks of one tile each, merged on the device."""
    _check(_dw("k", 5, 8, 2, 2, 700, d, kind, window=150, len_min=2))


@pytest.mark.parametrize("limit", [1, 2, 3, 7, 20])
@pytest.mark.parametrize("kind", [wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_CAUSAL_SLIDING])
def test_decode_long_shares(kind, limit):
    """A small grid: every CTA walks many tiles of several units (whole units in the middle of
    a share, partial ones at its ends), with the rescale, buffer-parity and merge paths."""
    _check(_dw("L", 4, 8, 2, 2, 1500, 128, kind, window=600, len_min=300), grid_limit=limit)


@pytest.mark.parametrize("limit", [1, 5])
@pytest.mark.parametrize("Hq,Hkv,S_q,d", [(8, 1, 1, 128), (32, 1, 1, 64), (16, 1, 4, 128)])
def test_decode_long_shares_row_widths(Hq, Hkv, S_q, d, limit):
    _check(_dw("Lr", 3, Hq, Hkv, S_q, 1100, d, wl.MASK_CAUSAL, len_min=S_q + 200), grid_limit=limit)


def test_decode_long_shares_sharp_rescale():
    """Long shares with sharpening scores, so rows rescale many times within one CTA."""
    w = _dw("sL", 2, 8, 2, 1, 3000, 128, wl.MASK_CAUSAL, len_min=2500)
    Qc, Kc, Vc, lens = wl.make_decode_inputs(w, stale_fill=float("nan"))
    Qc = (Qc.float() * 30).to(torch.bfloat16)
    Kc[:, :, :, :] = Kc.float() * torch.linspace(0.2, 2.0, 3000)[None, None, :, None]
    for b, L in enumerate(lens):
        Kc[b, :, L:] = float("nan")
    outs, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), lens, grid_limit=3)
    O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens, w.scale, w.kind)
    _compare(*outs[0], O_ref, L_ref)


@pytest.mark.parametrize("Hq,Hkv,S_q", [(8, 8, 1), (8, 1, 1), (16, 2, 2), (32, 1, 1), (8, 2, 8), (64, 1, 1),
                                        (8, 8, 7)])
def test_decode_packed_row_widths(Hq, Hkv, S_q):
    """group * S_q from 1 to 64 packed rows (16-, 32- and 64-column tiles)."""
    _check(_dw("r", 3, Hq, Hkv, S_q, 520, 128, wl.MASK_CAUSAL, len_min=S_q))


@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 256, 257])
def test_decode_cache_length_edges(L):
    """Cache lengths at and around tile edges, down to a single cached position."""
    w = _dw("e", 1, 4, 1, 1, 300, 128, wl.MASK_CAUSAL)
    Qc, Kc, Vc, _ = wl.make_decode_inputs(w.with_(S_cap=300), stale_fill=float("nan"))
    Kc[:, :, L:] = float("nan")
    Vc[:, :, L:] = float("nan")
    outs, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), [L])
    O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), [L], w.scale, w.kind)
    _compare(*outs[0], O_ref, L_ref)


@pytest.mark.parametrize("w_", [0, 1, 127, 128, 129, 300])
def test_decode_sliding_windows(w_):
    _check(_dw("w", 2, 8, 2, 3, 900, 64, wl.MASK_CAUSAL_SLIDING, window=w_, len_min=3))


def test_cross_attention_more_decoder_rows_than_encoder_positions():
    """FULL mask with encoder lengths shorter than the 32 decoder rows."""
    w = _dw("c", 3, 2, 2, 32, 64, 64, wl.MASK_FULL)
    Qc, Kc, Vc, _ = wl.make_decode_inputs(w)
    lens = [1, 17, 64]
    for b, L in enumerate(lens):
        Kc[b, :, L:] = float("nan")
        Vc[b, :, L:] = float("nan")
    outs, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), lens)
    O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens, w.scale, w.kind)
    _compare(*outs[0], O_ref, L_ref)


def test_decode_sharp_scores_rescale():
    """Query rows scaled by 30 so the running max jumps between tiles (the lazy rescale path)."""
    w = _dw("s", 2, 8, 2, 1, 1500, 128, wl.MASK_CAUSAL, len_min=900)
    Qc, Kc, Vc, lens = wl.make_decode_inputs(w, stale_fill=float("nan"))
    Qc = (Qc.float() * 30).to(torch.bfloat16)
    Kc[:, :, :, :] = Kc.float() * torch.linspace(0.2, 1.5, 1500)[None, None, :, None]
    for b, L in enumerate(lens):
        Kc[b, :, L:] = float("nan")
    outs, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), lens)
    O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens, w.scale, w.kind)
    _compare(*outs[0], O_ref, L_ref)


def test_decode_repeated_calls_are_identical():
    _check(_dw("rep", 4, 16, 2, 1, 2000, 128, wl.MASK_CAUSAL, len_min=500), reps=3)


def test_decode_step_equals_prefill_row():
    """One decode step over a full cache gives the prefill kernel's last row (to the bf16 bound)."""
    import transformer_self_attention_gb300 as tsa
    S, d = 600, 128
    w = wl.Workload("p", 1, 8, 2, S, d, "bf16", wl.MASK_CAUSAL, seed=5)
    Q, K, V = (t.cuda() for t in wl.make_inputs(w))
    O_pre, L_pre = tsa.Attention(1, 8, 2, S, d, kind=wl.MASK_CAUSAL)(Q, K, V)
    dec = tsa.DecodeAttention(1, 8, 2, 1, S, d, kind=wl.MASK_CAUSAL)
    O_dec, L_dec = dec(Q[:, :, S - 1:].contiguous(), K, V, [S])
    torch.cuda.synchronize()
    assert (O_dec.float() - O_pre[:, :, S - 1:].float()).abs().max().item() <= 2 * BF16_MAX_ABS
    assert (L_dec - L_pre[:, :, S - 1:]).abs().max().item() <= 2 * LSE_ABS


@pytest.mark.parametrize("w", wl.DECODE_ALL, ids=lambda w: w.name)
def test_decode_workloads_full_size(w):
    """The decode workloads at full size, every output against the oracle."""
    _check(w)


def _check_mode(w, mode, grid_limit=None):
    import transformer_self_attention_gb300 as tsa
    plan = tsa.DecodeAttention(w.B, w.Hq, w.Hkv, w.S_q, w.S_cap, w.d, scale=w.scale, kind=w.kind, window=w.window)
    plan.set_merge_mode(mode)
    Qc, Kc, Vc, lens = wl.make_decode_inputs(w, stale_fill=float("nan"))
    outs, _ = _run(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), lens, plan=plan, grid_limit=grid_limit)
    O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens, w.scale,
                                 w.kind, w.window)
    _compare(*outs[0], O_ref, L_ref)
    return outs[0]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("Hq,Hkv,S_q,d,kind", [(32, 1, 1, 128, wl.MASK_CAUSAL), (16, 16, 32, 64, wl.MASK_FULL),
                                               (32, 8, 4, 128, wl.MASK_CAUSAL_SLIDING), (8, 2, 2, 64, wl.MASK_CAUSAL)])
def test_decode_merge_modes_many_partials(Hq, Hkv, S_q, d, kind, mode):
    """Few units over every multiprocessor: each unit is split into many partials, merged by the
    last CTA to finish (mode 1) or by the merge kernel (mode 2)."""
    _check_mode(_dw("m", 2, Hq, Hkv, S_q, 3000, d, kind, window=700, len_min=S_q + 1500), mode)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("limit", [2, 7])
def test_decode_merge_modes_long_shares(limit, mode):
    _check_mode(_dw("ml", 4, 8, 2, 2, 1500, 128, wl.MASK_CAUSAL, len_min=300), mode, grid_limit=limit)


@pytest.mark.parametrize("w", [wl.DECODE_MQA_16K, wl.CROSS_MHA_4K], ids=lambda w: w.name)
def test_decode_merge_modes_agree_full_size(w):
    """Both merges of the same partials, against the oracle and against each other."""
    O1, L1 = _check_mode(w, 1)
    O2, L2 = _check_mode(w, 2)
    # the same partials summed in another order: at most a bf16 rounding apart (0.0078 near 1)
    assert np.abs(O1.astype(np.float64) - O2).max() <= BF16_MAX_ABS
    assert np.abs(L1.astype(np.float64) - L2).max() <= 1e-4


def test_decode_merge_mode_rejects_unknown_modes():
    import transformer_self_attention_gb300 as tsa
    plan = tsa.DecodeAttention(1, 2, 1, 1, 256, 64)
    for bad in (-1, 3):
        with pytest.raises(tsa.AttnError):
            plan.set_merge_mode(bad)


def test_decode_launch_count_follows_the_merge():
    """One kernel per call, two when the split units go to the merge kernel."""
    import transformer_self_attention_gb300 as tsa
    w = wl.DECODE_MQA_16K
    Qc, Kc, Vc, lens = wl.make_decode_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    plan = tsa.DecodeAttention(w.B, w.Hq, w.Hkv, w.S_q, w.S_cap, w.d, scale=w.scale, kind=w.kind, window=w.window)
    assert plan.launch_count() == 0
    for mode, n in ((1, 1), (2, 2), (0, 2)):  # this workload splits units over several CTAs
        plan.set_merge_mode(mode)
        _run(w, Q, K, V, lens, plan=plan)
        assert plan.launch_count() == n
    # no unit split (one tile per unit, as many CTAs as units): no merge kernel
    wt = _dw("one", 2, 4, 2, 1, 100, 64, wl.MASK_CAUSAL, len_min=50)
    Qt, Kt, Vt, lt = wl.make_decode_inputs(wt, stale_fill=float("nan"))
    outs, pt = _run(wt, Qt.cuda(), Kt.cuda(), Vt.cuda(), lt)
    assert pt.launch_count() == 1
    O_ref, L_ref = oracle.decode(Qt.float().numpy(), Kt.float().numpy(), Vt.float().numpy(), lt, wt.scale, wt.kind)
    _compare(*outs[0], O_ref, L_ref)


@pytest.mark.parametrize("mode", [0, 1])
def test_decode_back_to_back_calls_without_sync(mode):
    """Three steps enqueued on one handle before any synchronisation, each with its own query rows
    and lengths: every step's merge reads its own partials (the merge kernel waits for its decode
    grid, and the next decode grid for that merge), and every output matches the oracle."""
    import transformer_self_attention_gb300 as tsa
    w = _dw("b2b", 4, 32, 1, 1, 6000, 128, wl.MASK_CAUSAL, len_min=3000)
    plan = tsa.DecodeAttention(w.B, w.Hq, w.Hkv, w.S_q, w.S_cap, w.d, scale=w.scale, kind=w.kind)
    plan.set_merge_mode(mode)
    steps = []
    for k in range(3):
        Qc, Kc, Vc, lens = wl.make_decode_inputs(w.with_(seed=40 + k), stale_fill=float("nan"))
        Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
        O = torch.full_like(Q, float("nan"))
        LSE = torch.full((w.B, w.Hq, w.S_q), float("nan"), dtype=torch.float32, device=Q.device)
        plan(Q, K, V, lens, O=O, LSE=LSE)
        steps.append((Qc, Kc, Vc, lens, O, LSE, (Q, K, V)))
    torch.cuda.synchronize()
    st, code = plan.poll_device_error()
    assert st == 0 and code == 0
    assert plan.launch_count() == (2 if mode == 0 else 1)
    for Qc, Kc, Vc, lens, O, LSE, _ in steps:
        O_ref, L_ref = oracle.decode(Qc.float().numpy(), Kc.float().numpy(), Vc.float().numpy(), lens, w.scale,
                                     w.kind)
        _compare(O.float().cpu().numpy(), LSE.cpu().numpy(), O_ref, L_ref)
