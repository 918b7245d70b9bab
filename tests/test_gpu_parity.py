"""CUDA path vs the fp64 oracle, element by element (GPU).

Small shapes compare every output.  The five full-size workloads run in the
launch configuration bench.py times: the tiny fp32 workload, the causal 4K,
the 16K sliding-window and the local + global 8K workloads compare every output
(O and LSE over the whole tensor) with the oracle; the 32K causal GQA workload
(2,097,152 rows, about 6 minutes of oracle time on 16 host cores) compares a
stratified 1/16 of its rows -- 8 seeded rows out of every 128-row query tile of
every (batch, head) -- and checks properties over every output (finite, and
every output row inside the value range of its key/value head).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import all_rows, compare, gather_rows, oracle_rows, run_cuda, small, stratified_rows

pytestmark = pytest.mark.gpu

K_ALL = (wl.MASK_FULL, wl.MASK_CAUSAL, wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING, wl.MASK_LOCAL_GLOBAL)


def _full_compare(w):
    Qc, Kc, Vc = wl.make_inputs(w)
    O, LSE, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    bb, aa, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(w.S), indexing="ij")
    rows = np.stack([bb.ravel(), aa.ravel(), ii.ravel()], axis=1)
    O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, rows)
    return compare(w, O.float().cpu().numpy().reshape(-1, w.d), LSE.cpu().numpy().ravel(), O_ref, L_ref)


# ------------------------------------------------------------------ small shapes, every output

@pytest.mark.parametrize("S", [1, 127, 128, 129, 300])
@pytest.mark.parametrize("kind", K_ALL)
def test_bf16_d128_kinds_and_ragged_lengths(kind, S):
    G = sorted({0, S // 2, S - 1}) if kind == wl.MASK_LOCAL_GLOBAL else ()
    _full_compare(small("s", 1, 2, 2, S, 128, "bf16", kind, window=37, globals_idx=G))


@pytest.mark.parametrize("S", [1, 63, 64, 65, 127, 129, 191, 193, 300])
@pytest.mark.parametrize("kind", K_ALL)
def test_bf16_d64_kinds_and_ragged_lengths(kind, S):
    """d = 64 runs 64-key tiles (four CTAs per SM): lengths on both sides of 64-key boundaries, the
    band trimmed to the rows' interval, FULL decided per warp."""
    G = sorted({0, S // 2, S - 1}) if kind == wl.MASK_LOCAL_GLOBAL else ()
    _full_compare(small("s64", 1, 2, 2, S, 64, "bf16", kind, window=37, globals_idx=G))


@pytest.mark.parametrize("w_", [0, 31, 63, 64, 65, 191, 192])
@pytest.mark.parametrize("kind", [wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING, wl.MASK_LOCAL_GLOBAL])
def test_bf16_d64_windows_straddling_64_key_edges(kind, w_):
    G = (0, 200, 449) if kind == wl.MASK_LOCAL_GLOBAL else ()
    _full_compare(small("w64", 1, 2, 1, 450, 64, "bf16", kind, window=w_, globals_idx=G))


def test_bf16_d64_sharp_softmax_triggers_rescale():
    """Scores growing along the row force the lazy O rescale on many 64-key tiles."""
    w = small("sharp64", 1, 2, 2, 1000, 64, "bf16", wl.MASK_CAUSAL)
    Qc, Kc, Vc = wl.make_inputs(w)
    ramp = torch.linspace(0, 6, w.S).view(1, 1, w.S, 1)
    Kc = (Kc.float() + ramp * Qc.float().mean(dim=2, keepdim=True).sign()).to(torch.bfloat16)
    Qc = (Qc.float() * 3).to(torch.bfloat16)
    O, LSE, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, all_rows(w))
    compare(w, *gather_rows(O, LSE), O_ref, L_ref)


def test_bf16_d64_window_zero_returns_own_value_row():
    """w = 0 with 64-key tiles: each row sees only itself, so O_i = v_i exactly."""
    w = small("w0_64", 1, 2, 2, 300, 64, "bf16", wl.MASK_SLIDING, window=0)
    Qc, Kc, Vc = wl.make_inputs(w)
    O, LSE, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    assert torch.equal(O.cpu(), Vc)


@pytest.mark.parametrize("Hkv", [1, 2, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_gqa_and_mqa(Hkv, d):
    _full_compare(small("g", 2, 8, Hkv, 257, d, "bf16", wl.MASK_CAUSAL))


@pytest.mark.parametrize("w_", [0, 1, 127, 128, 129, 255])
@pytest.mark.parametrize("kind", [wl.MASK_SLIDING, wl.MASK_CAUSAL_SLIDING])
def test_bf16_windows_straddling_tile_edges(kind, w_):
    _full_compare(small("w", 1, 2, 1, 520, 64, "bf16", kind, window=w_))


@pytest.mark.parametrize("G", [[0], [519], [127, 128], [0, 1, 2, 3, 255, 256, 400], list(range(0, 520, 5))])
def test_bf16_local_global_placements(G):
    _full_compare(small("lg", 1, 3, 3, 520, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=40, globals_idx=G))


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_local_global_every_position_global(d):
    """Every position is a global token: every row sees every key (the full mask); the band items
    store no row and the global-row items, in key chunks, compute all of them."""
    w = small("lgall", 1, 2, 2, 300, d, "bf16", wl.MASK_LOCAL_GLOBAL, window=5, globals_idx=tuple(range(300)))
    Qc, Kc, Vc = wl.make_inputs(w)
    O, LSE, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    O_ref, L_ref = oracle_rows(w.with_(kind=wl.MASK_FULL, globals_idx=()), Qc, Kc, Vc, all_rows(w))
    compare(w, *gather_rows(O, LSE), O_ref, L_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_local_global_whole_global_tile(d):
    """A whole 128-position tile of global tokens (a full gathered key tile, a full global-row tile)."""
    _full_compare(small("lgt", 1, 2, 1, 520, d, "bf16", wl.MASK_LOCAL_GLOBAL, window=10,
                        globals_idx=tuple(range(128, 256))))


def test_bf16_local_global_globals_beyond_one_64_key_tile():
    """d = 64 (64-key tiles): 100 globals outside a query tile's band need two gathered key tiles."""
    G = list(range(2, 1000, 10))
    _full_compare(small("lg64g", 1, 2, 1, 1000, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=30, globals_idx=G))


def test_bf16_local_global_many_globals():
    """More than one gathered tile of global tokens (129 globals)."""
    _full_compare(small("lg2", 1, 2, 1, 700, 128, "bf16", wl.MASK_LOCAL_GLOBAL, window=9,
                        globals_idx=list(range(3, 700, 5))[:129]))


def test_local_global_repeated_calls_merge_every_time():
    """One handle, three calls with other inputs: the chunk counters of the global rows return to
    zero after every call (two global-row tiles, chunked keys, two gathered key tiles)."""
    G = sorted(set(range(2, 900, 4)) | {899})  # 226 globals
    w = small("lgrep", 1, 2, 1, 900, 64, "bf16", wl.MASK_LOCAL_GLOBAL, window=20, globals_idx=G)
    items, n_first = tsa_schedule(w)
    assert 1 + max(int(it[7]) for it in items[n_first:]) > 1 and max(int(it[7]) for it in items[:n_first]) == 2
    plan = None
    for seed in (5, 6, 7):
        ww = w.with_(seed=seed)
        Qc, Kc, Vc = wl.make_inputs(ww)
        O, LSE, plan = run_cuda(ww, Qc.cuda(), Kc.cuda(), Vc.cuda(), plan=plan)
        O_ref, L_ref = oracle_rows(ww, Qc, Kc, Vc, all_rows(ww))
        compare(ww, *gather_rows(O, LSE), O_ref, L_ref)


def tsa_schedule(w):
    import transformer_self_attention_gb300 as tsa
    return tsa.attn_schedule_host(w.B, w.Hq, w.Hkv, w.S, w.kind, w.window, list(w.globals_idx))


@pytest.mark.parametrize("kind", K_ALL)
@pytest.mark.parametrize("S", [1, 100, 257])
def test_f32_path_kinds(kind, S):
    G = sorted({0, S - 1}) if kind == wl.MASK_LOCAL_GLOBAL else ()
    _full_compare(small("f", 1, 4, 2, S, 64, "f32", kind, window=19, globals_idx=G))


def test_f32_d128():
    _full_compare(small("f128", 2, 2, 1, 200, 128, "f32", wl.MASK_CAUSAL))


def test_window_zero_returns_own_value_row():
    """w = 0: each row sees only itself, so O_i = v_i and LSE_i = s_ii."""
    w = small("w0", 1, 2, 2, 300, 128, "bf16", wl.MASK_SLIDING, window=0)
    Qc, Kc, Vc = wl.make_inputs(w)
    O, LSE, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    assert torch.equal(O.cpu(), Vc)
    s_ii = (Qc.double() * Kc.double()).sum(-1) * w.scale
    assert torch.allclose(LSE.cpu().double(), s_ii, atol=1e-3)


def test_sharp_softmax_triggers_rescale():
    """Scores growing along the row force the lazy O rescale on many tiles."""
    w = small("sharp", 1, 2, 2, 1024, 128, "bf16", wl.MASK_CAUSAL)
    Qc, Kc, Vc = wl.make_inputs(w)
    ramp = torch.linspace(0, 6, w.S).view(1, 1, w.S, 1)
    Kc = (Kc.float() + ramp * Qc.float().mean(dim=2, keepdim=True).sign()).to(torch.bfloat16)
    Qc = (Qc.float() * 3).to(torch.bfloat16)
    O, LSE, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    bb, aa, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(w.S), indexing="ij")
    rows = np.stack([bb.ravel(), aa.ravel(), ii.ravel()], axis=1)
    O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, rows)
    compare(w, O.float().cpu().numpy().reshape(-1, w.d), LSE.cpu().numpy().ravel(), O_ref, L_ref)


def test_handle_reuse_and_distinct_buffers():
    w = small("reuse", 1, 4, 2, 384, 128, "bf16", wl.MASK_CAUSAL)
    Qc, Kc, Vc = wl.make_inputs(w)
    O1, L1, plan = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    w2 = w.with_(seed=99)
    Q2, K2, V2 = wl.make_inputs(w2)
    O2, L2, _ = run_cuda(w2, Q2.cuda(), K2.cuda(), V2.cuda(), plan=plan)
    O1b, L1b, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda(), plan=plan)
    assert torch.equal(O1, O1b) and torch.equal(L1, L1b)
    assert not torch.equal(O1, O2)


# ------------------------------------------------------------------ the five workloads

def test_tiny_full_f32_every_output():
    w = wl.TINY_FULL_F32
    Qc, Kc, Vc = wl.make_inputs(w)
    O, LSE, _ = run_cuda(w, Qc.cuda(), Kc.cuda(), Vc.cuda())
    O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, all_rows(w))
    compare(w, *gather_rows(O, LSE), O_ref, L_ref, report=f"{w.name} (every row)")


def _value_range_holds(w, O, LSE, V):
    """Every output finite and inside the per-column value range of its kv head (the weights
    are a convex combination), over the whole tensor."""
    assert bool(torch.isfinite(O).all()) and bool(torch.isfinite(LSE).all())
    g = w.Hq // w.Hkv
    vmax = V.float().amax(dim=2).repeat_interleave(g, dim=1)  # [B, Hq, d]
    vmin = V.float().amin(dim=2).repeat_interleave(g, dim=1)
    assert bool((O.float() <= vmax[:, :, None, :] + 2e-2).all())
    assert bool((O.float() >= vmin[:, :, None, :] - 2e-2).all())


@pytest.mark.parametrize("w", [wl.CAUSAL_MHA_4K, wl.SWA_GQA_16K, wl.LONGFORMER_8K], ids=lambda w: w.name)
def test_full_size_workload_every_output(w):
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    O, LSE, _ = run_cuda(w, Q, K, V)
    _value_range_holds(w, O, LSE, V)
    O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, all_rows(w))
    compare(w, *gather_rows(O, LSE), O_ref, L_ref, report=f"{w.name} (every row)")


def test_full_size_32k_stratified_sixteenth():
    w = wl.CAUSAL_GQA_32K
    Qc, Kc, Vc = wl.make_inputs(w)
    Q, K, V = Qc.cuda(), Kc.cuda(), Vc.cuda()
    O, LSE, _ = run_cuda(w, Q, K, V)
    _value_range_holds(w, O, LSE, V)
    rows = stratified_rows(w, per_tile=8)
    assert rows.shape[0] * 16 == w.B * w.Hq * w.S
    O_ref, L_ref = oracle_rows(w, Qc, Kc, Vc, rows)
    compare(w, *gather_rows(O, LSE, rows), O_ref, L_ref, report=f"{w.name} (stratified 1/16 of rows)")
