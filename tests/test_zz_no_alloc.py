"""attn_forward_noalloc: the forward pass for callers that cannot allocate device memory.

Such callers (code inside a memory pool it does not own, runtimes that forbid
cudaMalloc after start-up, processes whose device footprint must stay fixed)
call one entry point whose scratch lives in a fixed library-owned device array.
These tests call it through the C ABI and compare its outputs with the fp64
oracle and with the handle-based attn_forward on two calls in a row, the second
with different inputs and global positions so stale scratch would show; they
read its error word through attn_forward_noalloc_poll_error, also after a wait
that was made to run out.  The file is named to be collected last; it also
passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import transformer_self_attention_gb300 as tsa
import workloads as wl
from gpu_util import BF16_MAX_ABS, BF16_REL_L2, LSE_ABS, all_rows, compare, gather_rows, oracle_rows, run_cuda, small

pytestmark = pytest.mark.gpu


def _noalloc(w, Q, K, V):
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device=Q.device)
    st = tsa.attn_forward_noalloc(w.B, w.Hq, w.Hkv, w.S, w.d, w.scale, w.kind, w.window, list(w.globals_idx),
                                  Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert st == tsa.ATTN_OK, tsa.attn_status_string(st)
    torch.cuda.synchronize()
    return O, LSE


def _close(w, O, LSE, O_ref, L_ref):
    a, b = O.double().cpu().numpy(), O_ref.double().cpu().numpy()
    assert np.all(np.isfinite(a)) and bool(torch.isfinite(LSE).all())
    assert np.max(np.abs(a - b)) <= BF16_MAX_ABS
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= BF16_REL_L2
    assert float((LSE - L_ref).abs().max()) <= LSE_ABS


@pytest.mark.parametrize("w", [
    small("na_causal", 1, 8, 2, 700, 128, "bf16", wl.MASK_CAUSAL),
    small("na_lg", 2, 4, 4, 600, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=33, globals_idx=(0, 5, 300, 599)),
    small("na_swa", 1, 4, 1, 520, 128, "bf16", wl.MASK_CAUSAL_SLIDING, window=129),
], ids=lambda w: w.name)
def test_noalloc_matches_oracle_and_attn_forward_on_two_calls(w):
    # second call: other inputs, and for local + global other global positions
    w2 = w.with_(seed=w.seed + 7, globals_idx=(1, 127, 128, 598) if w.globals_idx else ())
    for ww in (w, w2):
        Qc, Kc, Vc = wl.make_inputs(ww)
        Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
        O_ref, L_ref, plan = run_cuda(ww, Q, K, V)
        plan.close()
        O, LSE = _noalloc(ww, Q, K, V)
        O_or, L_or = oracle_rows(ww, Qc, Kc, Vc, all_rows(ww))
        compare(ww, *gather_rows(O, LSE), O_or, L_or)
        _close(ww, O, LSE, O_ref, L_ref)
    assert tsa.attn_forward_noalloc_poll_error() == (tsa.ATTN_OK, 0)


def test_noalloc_repeat_call_allocates_no_device_memory():
    w = small("na_mem", 1, 4, 4, 384, 128, "bf16", wl.MASK_LOCAL_GLOBAL, window=20, globals_idx=(3, 200))
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    O1, L1 = _noalloc(w, Q, K, V)           # first call on the device: module and symbol set-up
    free_before, _ = torch.cuda.mem_get_info()
    O2, L2 = _noalloc(w, Q, K, V)
    assert tsa.attn_forward_noalloc_poll_error() == (tsa.ATTN_OK, 0)
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_noalloc_error_word_reports_a_wait_that_ran_out():
    """The watchdog bits of this entry point are readable: a withheld V load makes a bounded wait
    run out; the poll returns ATTN_ERR_DEVICE_TIMEOUT with the role bits and clears the word, and
    the next call (local + global, with chunked global rows) is correct again."""
    w = small("na_wd", 1, 2, 2, 520, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=40, globals_idx=(0, 300))
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    assert tsa.attn_forward_noalloc_set_watchdog(50_000_000, 1) == tsa.ATTN_OK  # 50 ms, V withheld
    try:
        _noalloc(w, Q, K, V)
        st, code = tsa.attn_forward_noalloc_poll_error()
    finally:
        assert tsa.attn_forward_noalloc_set_watchdog(2_000_000_000, 0) == tsa.ATTN_OK
    assert st == tsa.ATTN_ERR_DEVICE_TIMEOUT and code != 0 and (code & ~7) == 0, (st, code)
    assert tsa.attn_forward_noalloc_poll_error() == (tsa.ATTN_OK, 0)  # cleared by the poll
    O, LSE = _noalloc(w, Q, K, V)
    O_or, L_or = oracle_rows(w, Qc, Kc, Vc, all_rows(w))
    compare(w, *gather_rows(O, LSE), O_or, L_or)
    assert tsa.attn_forward_noalloc_poll_error() == (tsa.ATTN_OK, 0)


def test_noalloc_rejects_problems_beyond_the_scratch_limit():
    # 8 x 64 heads x 512 query tiles = 262,144 work items of 32 bytes: 8 MiB of work list alone,
    # more than the 8 MiB array once the error word is counted
    st = tsa.attn_forward_noalloc(8, 64, 8, 65536, 128, 0.088, wl.MASK_CAUSAL, 0, [], 256, 256, 256, 256, 0, 0)
    assert st == tsa.ATTN_ERR_UNSUPPORTED
    assert tsa.NOALLOC_SCRATCH_BYTES == 8 << 20
    assert tsa.attn_forward_noalloc_set_watchdog(0, 0) == tsa.ATTN_ERR_INVALID_ARG
