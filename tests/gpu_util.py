"""Helpers of the GPU parity tests: run the CUDA path, run the oracle, compare."""
import numpy as np
import torch

import oracle
import workloads as wl

# Bounds the outputs must meet (bf16 inputs / fp32 inputs; LSE absolute).
BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 5e-3
F32_MAX_ABS, F32_REL_L2 = 1e-4, 1e-4
LSE_ABS = 1e-3


def run_cuda(w, Q, K, V, plan=None):
    """CUDA path through the C ABI; outputs NaN-poisoned first so unwritten rows show."""
    import transformer_self_attention_gb300 as tsa
    if plan is None:
        plan = tsa.Attention(w.B, w.Hq, w.Hkv, w.S, w.d, dtype=w.dtype, scale=w.scale, kind=w.kind,
                             window=w.window, global_idx=list(w.globals_idx))
    O = torch.full_like(Q, float("nan"))
    LSE = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device=Q.device)
    plan(Q, K, V, O=O, LSE=LSE)
    torch.cuda.synchronize()
    st, code = plan.poll_device_error()
    assert st == 0 and code == 0, f"device error word {code}"
    return O, LSE, plan


def oracle_rows(w, Qc, Kc, Vc, rows):
    """Oracle outputs for rows = array of (b, a, i)."""
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    Qn = Qc.float().numpy()
    qrows = Qn[rows[:, 0], rows[:, 1], rows[:, 2]]
    return oracle.attention_rows(Kc.float().numpy(), Vc.float().numpy(), w.Hq, w.scale, w.kind, w.window,
                                 list(w.globals_idx), qrows, rows[:, 0], rows[:, 1], rows[:, 2])


# Error norms of the comparisons that asked to be reported (name -> one line); the terminal
# summary of the test session prints them (tests/conftest.py).
REPORT = {}


def compare(w, O_gpu, LSE_gpu, O_ref, LSE_ref, report=None):
    """Assert the error bounds; returns (max_abs, rel_l2, lse_max_abs).

    The relative L2 error is taken over every row passed in: the whole tensor when the
    caller passes every row.  With ``report`` set, the norms are recorded under that name.
    """
    O_gpu = np.asarray(O_gpu, dtype=np.float64)
    LSE_gpu = np.asarray(LSE_gpu, dtype=np.float64)
    assert np.all(np.isfinite(O_gpu)), "non-finite (unwritten?) outputs"
    assert np.all(np.isfinite(LSE_gpu)), "non-finite LSE"
    diff = O_gpu - O_ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(O_ref), 1e-30))
    lse_err = float(np.max(np.abs(LSE_gpu - LSE_ref))) if LSE_ref.size else 0.0
    ma, rl = (BF16_MAX_ABS, BF16_REL_L2) if w.dtype == "bf16" else (F32_MAX_ABS, F32_REL_L2)
    if report:
        REPORT[report] = (f"rows {O_ref.shape[0]}  max-abs {max_abs:.3e}  rel-L2 {rel:.3e}  "
                          f"LSE max-abs {lse_err:.3e}")
    assert max_abs <= ma, f"max abs error {max_abs:.3e} > {ma}"
    assert rel <= rl, f"relative L2 error {rel:.3e} > {rl}"
    assert lse_err <= LSE_ABS, f"LSE error {lse_err:.3e} > {LSE_ABS}"
    return max_abs, rel, lse_err


def sample_rows(w, n_random=192, seed=0):
    """(b, a, i) rows: edges, tile boundaries, global rows, a window edge, and random rows."""
    rng = np.random.default_rng(seed)
    S, T = w.S, 128
    pos = {0, 1, S - 1, S - 2, min(T - 1, S - 1), min(T, S - 1), S // 2}
    pos |= {p for p in (w.window, w.window + 1, S - 1 - w.window) if 0 <= p < S}
    pos |= set(w.globals_idx)
    pos |= {min(S - 1, g + d) for g in w.globals_idx for d in (-1, 1) if g + d >= 0}
    rows = []
    for p in sorted(pos):
        for a in {0, w.Hq - 1, w.Hq // 2}:
            rows.append((int(rng.integers(w.B)), a, p))
    for _ in range(n_random):
        rows.append((int(rng.integers(w.B)), int(rng.integers(w.Hq)), int(rng.integers(S))))
    return np.array(rows, dtype=np.int64)


def all_rows(w):
    """Every (b, a, i) row of a workload, in the [B, Hq, S] order of O."""
    bb, aa, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(w.S), indexing="ij")
    return np.stack([bb.ravel(), aa.ravel(), ii.ravel()], axis=1).astype(np.int64)


def stratified_rows(w, per_tile=8, seed=0):
    """per_tile distinct seeded rows out of every 128-row query tile of every (b, a): 1/16 of
    all rows at per_tile = 8, and every (batch, head, query tile) is covered."""
    rng = np.random.default_rng(seed)
    T = 128
    out = []
    for b in range(w.B):
        for a in range(w.Hq):
            for t0 in range(0, w.S, T):
                n = min(T, w.S - t0)
                for r in rng.choice(n, size=min(per_tile, n), replace=False):
                    out.append((b, a, t0 + int(r)))
    return np.array(out, dtype=np.int64)


def gather_rows(O, LSE, rows=None):
    """GPU outputs of the listed rows (every row, in all_rows order, when rows is None), as
    float64 host arrays ([n, d], [n])."""
    if rows is None:
        return (O.float().cpu().numpy().reshape(-1, O.shape[-1]).astype(np.float64),
                LSE.cpu().numpy().ravel().astype(np.float64))
    r = torch.as_tensor(rows, device=O.device)
    return (O[r[:, 0], r[:, 1], r[:, 2]].float().cpu().numpy().astype(np.float64),
            LSE[r[:, 0], r[:, 1], r[:, 2]].cpu().numpy().astype(np.float64))


def small(name, B, Hq, Hkv, S, d, dtype, kind, window=0, globals_idx=(), seed=11):
    return wl.Workload(name, B, Hq, Hkv, S, d, dtype, kind, window=window, globals_idx=tuple(globals_idx),
                       seed=seed)
