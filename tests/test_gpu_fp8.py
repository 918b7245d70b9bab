"""E4M3 (FP8) inputs on the GPU vs the fp64 oracle over the dequantised values.

The oracle attends over q8 * dq, k8 * dk, v8 * dv exactly; the remaining difference is
the E4M3 rounding of P before the second product and fp32 accumulation.  Round to
nearest with 3 mantissa bits gives each weight a relative error of at most 2^-4, with a
standard deviation of about 2^-4 / sqrt(3) = 0.036.  The error of an output row,
sum_j delta_j p_j v_j / l, is bounded by 2^-4 * max|v| (all errors of one sign), and
relative to |O| it is largest where O is an average of many values that cancel (full
and wide-window rows).  Bounds: max-abs 0.15 (2^-4 times ~2.4, below the largest
value magnitudes) and relative L2 5e-2 (just under 2^-4).  LSE comes from the fp32
weights and keeps the bf16 path's 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import LSE_ABS, sample_rows, small

pytestmark = pytest.mark.gpu

FP8_MAX_ABS, FP8_REL_L2 = 0.15, 5e-2


def _run(w):
    import transformer_self_attention_gb300 as tsa
    Q8, K8, V8, (dq, dk, dv) = wl.make_fp8_inputs(w)
    plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype="e4m3", scale=w.scale, kind=w.kind, window=w.window)
    plan.set_fp8_descale(dq, dk, dv)
    O = torch.full((w.B, w.Hq, w.S, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    L = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device="cuda")
    plan(Q8.cuda(), K8.cuda(), V8.cuda(), O=O, LSE=L)
    torch.cuda.synchronize()
    assert plan.poll_device_error() == (0, 0)
    return O.float().cpu().numpy(), L.cpu().numpy(), (Q8, K8, V8, dq, dk, dv)


def _check(O, L, O_ref, L_ref):
    assert np.isfinite(O).all() and np.isfinite(L).all()
    d = O.astype(np.float64) - O_ref
    max_abs = float(np.abs(d).max())
    rel = float(np.linalg.norm(d) / np.linalg.norm(O_ref))
    lse = float(np.abs(L - L_ref).max())
    print(f"fp8 errors: max-abs {max_abs:.3e} rel-L2 {rel:.3e} LSE {lse:.3e}")
    assert max_abs <= FP8_MAX_ABS and rel <= FP8_REL_L2 and lse <= LSE_ABS, (max_abs, rel, lse)


@pytest.mark.parametrize("S", [1, 129, 300])
@pytest.mark.parametrize("kind", [wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING])
def test_fp8_kinds(kind, S):
    w = small("f8", 2, 4, 2, S, 128, "bf16", kind, window=37)
    O, L, (Q8, K8, V8, dq, dk, dv) = _run(w)
    O_ref, L_ref = oracle.attention(Q8.float().numpy(), K8.float().numpy(), V8.float().numpy(), w.scale * dq * dk,
                                    w.kind, w.window)
    _check(O, L, O_ref * dv, L_ref)


def test_fp8_full_size_causal_4k():
    w = wl.CAUSAL_MHA_4K
    O, L, (Q8, K8, V8, dq, dk, dv) = _run(w)
    rows = sample_rows(w, n_random=96)
    Qn = Q8.float().numpy()
    O_ref, L_ref = oracle.attention_rows(K8.float().numpy(), V8.float().numpy(), w.Hq, w.scale * dq * dk, w.kind,
                                         w.window, None, Qn[rows[:, 0], rows[:, 1], rows[:, 2]], rows[:, 0],
                                         rows[:, 1], rows[:, 2])
    _check(O[rows[:, 0], rows[:, 1], rows[:, 2]], L[rows[:, 0], rows[:, 1], rows[:, 2]], O_ref * dv, L_ref)


def test_fp8_unsupported_shapes():
    import transformer_self_attention_gb300 as tsa
    for kw in (dict(d=64, kind=wl.MASK_CAUSAL), dict(d=128, kind=wl.MASK_LOCAL_GLOBAL, global_idx=[0])):
        with pytest.raises(tsa.AttnError) as e:
            tsa.Attention(1, 2, 2, 256, kw["d"], dtype="e4m3", kind=kw["kind"], window=3,
                          global_idx=kw.get("global_idx"))
        assert e.value.status == tsa.ATTN_ERR_UNSUPPORTED
    plan = tsa.Attention(1, 2, 2, 256, 128, dtype="e4m3", kind=wl.MASK_CAUSAL)
    with pytest.raises(tsa.AttnError):
        plan.set_alibi([0.1, 0.2])
