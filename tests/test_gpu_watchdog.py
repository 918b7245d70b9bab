"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The test hook makes the producer never load V, so the MMA issuer's wait for V
runs out after the (short) limit.  The kernel must record the error in the
handle's error word, free its tensor memory and return; the context must stay
usable (a normal call afterwards gives correct results).
"""
import numpy as np
import pytest
import torch

import transformer_self_attention_gb300 as tsa
import workloads as wl
from gpu_util import compare, oracle_rows, run_cuda, small

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [128, 64])  # d = 64: the 64-key-tile kernel, four CTAs per SM
def test_withheld_load_times_out_and_context_survives(d):
    w = small("wd", 1, 2, 2, 256, d, "bf16", wl.MASK_CAUSAL)
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, kind=w.kind)
    plan.set_watchdog(50_000_000, withhold=1)  # 50 ms
    plan(Q, K, V)
    st, code = plan.poll_device_error()
    assert st == tsa.ATTN_ERR_DEVICE_TIMEOUT
    # bit 1 producer (waiting for V to be consumed), bit 2 MMA issuer (waiting for V to land);
    # whichever role's limit runs out first records its bit, the others abort on the shared flag
    assert code != 0 and (code & ~7) == 0, f"unexpected error word {code}"
    # the error word is cleared by the poll; the context is still usable
    plan.set_watchdog(2_000_000_000, withhold=0)
    O, LSE, _ = run_cuda(w, Q, K, V, plan=plan)
    bb, aa, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(w.S), indexing="ij")
    rows = np.stack([bb.ravel(), aa.ravel(), ii.ravel()], axis=1)
    O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, rows)
    compare(w, O.float().cpu().numpy().reshape(-1, w.d), LSE.cpu().numpy().ravel(), O_ref, L_ref)
    torch.cuda.synchronize()


def test_local_global_abort_keeps_the_chunk_counters_consistent():
    """Local + global with chunked global rows: every chunk item counts itself in even when its
    wait ran out, so the counters return to zero and the next call merges correctly."""
    w = small("wdlg", 1, 2, 2, 700, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=40, globals_idx=(0, 1, 350, 699))
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, kind=w.kind, window=w.window, global_idx=list(w.globals_idx))
    items, n_first = tsa.attn_schedule_host(w.B, w.Hq, w.Hkv, w.S, w.kind, w.window, list(w.globals_idx))
    assert 1 + max(int(it[7]) for it in items[n_first:]) > 1  # the global rows are chunked
    plan.set_watchdog(50_000_000, withhold=1)
    plan(Q, K, V)
    st, code = plan.poll_device_error()
    assert st == tsa.ATTN_ERR_DEVICE_TIMEOUT and code != 0
    plan.set_watchdog(2_000_000_000, withhold=0)
    for _ in range(2):
        O, LSE, _ = run_cuda(w, Q, K, V, plan=plan)
        bb, aa, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(w.S), indexing="ij")
        rows = np.stack([bb.ravel(), aa.ravel(), ii.ravel()], axis=1)
        O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, rows)
        compare(w, O.float().cpu().numpy().reshape(-1, w.d), LSE.cpu().numpy().ravel(), O_ref, L_ref)
