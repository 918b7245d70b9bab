"""The host tile schedule against brute force from the oracle's mask predicate (bit-exact).

For every listed key tile the schedule's class (FULL / PARTIAL) must equal the
oracle's enumerated class; unlisted tiles must be SKIP (for local + global: hold
no allowed pair outside the global rows and columns); and simulating what the
kernels evaluate from the work items -- FULL tiles whole, PARTIAL tiles through
the in-tile predicate, the gathered global keys outside a tile's band, the dense
global-row chunks -- must count exactly the allowed pairs of every row, each once.
"""
import numpy as np
import pytest

import oracle
import transformer_self_attention_gb300 as tsa
import workloads as wl

T = tsa.TILE


def _kernel_interval(kind, i, S, w):
    """The per-row key interval the kernels use on PARTIAL tiles (before global columns)."""
    lo = np.zeros_like(i)
    hi = np.full_like(i, S - 1)
    if kind == tsa.MASK_CAUSAL:
        hi = i.copy()
    elif kind == tsa.MASK_CAUSAL_SLIDING:
        lo, hi = i - w, i.copy()
    elif kind in (tsa.MASK_SLIDING, tsa.MASK_LOCAL_GLOBAL):
        lo, hi = i - w, i + w
    return lo, np.minimum(hi, S - 1)


def _simulate(items, n_first, kind, S, w, G, check_classes=True):
    """Per-row count of the pairs the kernels evaluate as allowed, for batch-head 0."""
    isg = np.zeros(S, dtype=bool)
    isg[list(G)] = True
    Garr = np.array(sorted(G), dtype=np.int64)
    counts = np.zeros(S, dtype=np.int64)
    classes = oracle.tile_classes(kind, S, w, list(G)) if check_classes else None
    lg = kind == tsa.MASK_LOCAL_GLOBAL
    seen_tiles = set()
    chunks = {}
    for n, it in enumerate(items):
        bh, qt, kb, ke, fb, fe, flags, ngt = (int(x) for x in it)
        if bh != 0:
            continue
        if flags & tsa.WORK_GLOBAL_ROWS:
            # one key chunk [kb, ke) of the dense pass over the gathered global rows
            assert n >= n_first
            rows = Garr[qt * T:(qt + 1) * T]
            nk = (S + T - 1) // T
            assert 0 <= kb <= fb <= fe <= ke <= nk
            assert fe <= S // T                        # FULL only for whole key tiles
            assert ke - fe <= 1 and (fe == ke or ke == nk)
            chunks.setdefault(qt, []).append((ngt, kb, ke))
            counts[rows] += min(ke * T, S) - kb * T
            continue
        assert n < n_first
        assert (qt not in seen_tiles), "query tile listed twice"
        seen_tiles.add(qt)
        i = np.arange(qt * T, min(S, (qt + 1) * T))
        lo, hi = _kernel_interval(kind, i, S, w)
        keep = ~isg[i] if lg else np.ones(i.size, dtype=bool)
        assert kb <= fb <= fe <= ke
        for t in range(kb, ke):
            j = np.arange(t * T, min(S, (t + 1) * T))
            full = fb <= t < fe
            if check_classes:
                assert classes[qt, t] == (1 if full else 2), (qt, t, classes[qt, t], full)
            if full:
                counts[i[keep]] += j.size
            else:
                ok = ((j[None, :] >= lo[:, None]) & (j[None, :] <= hi[:, None]))
                if lg:
                    ok |= isg[j][None, :]
                counts[i[keep]] += ok[keep].sum(axis=1)
        if check_classes and not lg:
            for t in set(range(classes.shape[1])) - set(range(kb, ke)):
                assert classes[qt, t] == 0, (qt, t)
        n_out = int(((Garr < kb * T) | (Garr >= ke * T)).sum()) if lg else 0
        assert bool(flags & tsa.WORK_GLOBAL_COLS) == (n_out > 0)
        assert bool(flags & tsa.WORK_HAS_GLOBAL_ROWS) == bool(lg and isg[i].any())
        if flags & tsa.WORK_GLOBAL_COLS:
            # the gathered tiles hold exactly the global keys outside the band, every one allowed
            assert lg and ngt == (n_out + T - 1) // T
            counts[i[keep]] += n_out
    assert seen_tiles == set(range((S + T - 1) // T))
    nk = (S + T - 1) // T
    for qt, cs in chunks.items():  # the chunks of each gathered row tile cover [0, nk) once, in order
        cs.sort()
        assert [c for c, _, _ in cs] == list(range(len(cs)))
        assert cs[0][1] == 0 and cs[-1][2] == nk
        assert all(cs[k][2] == cs[k + 1][1] for k in range(len(cs) - 1))
    return counts


def _check(kind, S, w=0, G=(), B=1, Hq=2, Hkv=1, check_classes=True):
    items, n_first = tsa.attn_schedule_host(B, Hq, Hkv, S, kind, w, list(G))
    nq = (S + T - 1) // T
    assert n_first == B * Hq * nq
    if kind == tsa.MASK_LOCAL_GLOBAL and G:
        n_chunks = 1 + max(int(it[7]) for it in items[n_first:])
        assert len(items) - n_first == B * Hq * ((len(G) + T - 1) // T) * n_chunks
    else:
        assert len(items) == n_first
    # every (bh, q_tile) exactly once among the first-launch items
    pairs = {(int(a), int(b)) for a, b in items[:n_first, :2]}
    assert pairs == {(bh, q) for bh in range(B * Hq) for q in range(nq)}
    # kv-head groups whose K and V fit in 32 MB (at d = 128) one after another when every group holds
    # at least 4096 items, longest first in each
    cost = (items[:n_first, 3] - items[:n_first, 2]) + items[:n_first, 7]
    g_kv = max(1, min(B * Hkv, (32 << 20) // (512 * S)))
    if g_kv * (Hq // Hkv) * nq < 4096:  # short problems: longest first over all heads
        g_kv = B * Hkv
    bh = items[:n_first, 0]
    unit = (bh // Hq) * Hkv + (bh % Hq) // (Hq // Hkv)
    gidx = unit // g_kv
    assert np.all(np.diff(gidx) >= 0)
    for g in np.unique(gidx):
        assert np.all(np.diff(cost[gidx == g]) <= 0)
    if len(items) > n_first:  # global-row chunks are no longer than the longest query-tile item
        assert np.all(items[n_first:, 3] - items[n_first:, 2] <= max(1, int(cost.max())))
    counts = _simulate(items, n_first, kind, S, w, set(G), check_classes)
    expect = oracle.row_counts(kind, S, w, list(G))
    assert np.array_equal(counts, expect)


SWEEP_S = [1, 2, 127, 128, 129, 300, 515]


@pytest.mark.parametrize("S", SWEEP_S)
@pytest.mark.parametrize("kind", [tsa.MASK_FULL, tsa.MASK_CAUSAL])
def test_schedule_dense_kinds(kind, S):
    _check(kind, S)


@pytest.mark.parametrize("S", SWEEP_S)
@pytest.mark.parametrize("w", [0, 1, 3, 127, 128, 129, 200, 600])
@pytest.mark.parametrize("kind", [tsa.MASK_SLIDING, tsa.MASK_CAUSAL_SLIDING])
def test_schedule_window_kinds(kind, S, w):
    _check(kind, S, w)


@pytest.mark.parametrize("S,w,G", [
    (1, 0, [0]), (129, 3, [0]), (129, 3, [128]), (300, 5, [0, 127, 128, 299]), (300, 0, []),
    (515, 60, [3, 4, 5, 200, 511, 514]), (515, 300, [0, 100]), (700, 1, list(range(0, 700, 3))),
    (1000, 128, [127, 128, 255, 256, 999]),
])
def test_schedule_local_global(S, w, G):
    _check(tsa.MASK_LOCAL_GLOBAL, S, w, G)


@pytest.mark.parametrize("w", [wl.TINY_FULL_F32, wl.CAUSAL_MHA_4K, wl.SWA_GQA_16K, wl.LONGFORMER_8K],
                         ids=lambda w: w.name)
def test_schedule_workloads(w):
    _check(w.kind, w.S, w.window, w.globals_idx, B=1, Hq=2, Hkv=1)


def test_schedule_long_causal_classes():
    """The 32K causal workload: classes only (the coverage follows for interval masks)."""
    w = wl.CAUSAL_GQA_32K
    items, n_first = tsa.attn_schedule_host(1, 1, 1, w.S, w.kind, 0, [])
    classes = oracle.tile_classes(w.kind, w.S, 0, [])
    got = np.zeros_like(classes)
    for it in items:
        _, qt, kb, ke, fb, fe, _, _ = (int(x) for x in it)
        for t in range(kb, ke):
            got[qt, t] = 1 if fb <= t < fe else 2
    assert np.array_equal(got, classes)


def test_schedule_heads_and_batches():
    items, n_first = tsa.attn_schedule_host(3, 8, 2, 300, tsa.MASK_CAUSAL, 0, [])
    per_bh = {}
    for it in items:
        per_bh.setdefault(int(it[0]), []).append(tuple(int(x) for x in it[1:]))
    ref = sorted(per_bh[0])
    assert sorted(per_bh) == list(range(24))
    assert all(sorted(v) == ref for v in per_bh.values())


def test_duplicate_globals_are_removed():
    a, _ = tsa.attn_schedule_host(1, 1, 1, 300, tsa.MASK_LOCAL_GLOBAL, 5, [7, 7, 250, 7])
    b, _ = tsa.attn_schedule_host(1, 1, 1, 300, tsa.MASK_LOCAL_GLOBAL, 5, [7, 250])
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ backward key-tile schedule

@pytest.mark.parametrize("S", [1, 127, 128, 129, 300, 515])
@pytest.mark.parametrize("kind,w", [(tsa.MASK_FULL, 0), (tsa.MASK_CAUSAL, 0), (tsa.MASK_SLIDING, 3),
                                    (tsa.MASK_SLIDING, 130), (tsa.MASK_CAUSAL_SLIDING, 0),
                                    (tsa.MASK_CAUSAL_SLIDING, 200)])
def test_kv_schedule_matches_brute_force(kind, S, w):
    """Every key tile once; its query-tile range holds exactly the tiles with an allowed pair, and
    its FULL range exactly the tiles the oracle's enumeration calls FULL (transposed classes)."""
    items = tsa.attn_kv_schedule_host(S, kind, w)
    nk = (S + T - 1) // T
    assert sorted(int(x) for x in items[:, 0]) == list(range(nk))
    classes = oracle.tile_classes(kind, S, w, [])  # [q tile, k tile]
    for kt, qb, qe, fb, fe, *_ in (tuple(int(x) for x in it) for it in items):
        for qt in range(classes.shape[0]):
            c = classes[qt, kt]
            if qb <= qt < qe:
                assert c == (1 if fb <= qt < fe else 2), (kt, qt, c)
            else:
                assert c == 0, (kt, qt)
    lengths = items[:, 2] - items[:, 1]
    assert np.all(np.diff(lengths) <= 0)


def _lg_bwd_kernel_counts(S, w, G, lst, off):
    """Per row (dQ view: a thread per query row over its list's key tiles) the pairs the
    backward kernels evaluate as allowed: FULL entries whole, the others through the kernel's
    bit mask (window interval, the interval [0, S - 1] for a global row, the tile's global
    columns).  The mask is symmetric and the dK/dV kernel runs the same predicate with rows and
    columns swapped, so the same counts hold per key column."""
    isg = np.zeros(S, dtype=bool)
    isg[list(G)] = True
    counts = np.zeros(S, dtype=np.int64)
    for i in range(S):
        x = i // T
        lo, hi = max(0, i - w), min(S - 1, i + w)
        if isg[i]:
            lo, hi = 0, S - 1
        for e in lst[off[x]:off[x + 1]]:
            t = int(e) & (tsa.LIST_FULL - 1)
            cols = np.arange(t * T, t * T + T)
            if int(e) & tsa.LIST_FULL:
                counts[i] += T
                continue
            inside = cols < S
            ok = ((cols >= lo) & (cols <= hi)) | (isg[np.minimum(cols, S - 1)] & inside)
            counts[i] += int(np.count_nonzero(ok & inside))
    return counts


@pytest.mark.parametrize("S,w,G", [(1, 0, (0,)), (127, 3, (0, 126)), (128, 5, (64,)), (129, 0, (128,)),
                                   (300, 40, (0, 100, 299)), (520, 130, (0, 127, 128, 255, 519)),
                                   (700, 200, ()), (640, 63, tuple(range(0, 640, 5))),
                                   (520, 10, tuple(range(128, 256))), (640, 3, tuple(range(0, 128)) + (600,))])
def test_lg_backward_lists_match_brute_force(S, w, G):
    """Local + global backward lists against the oracle's enumeration: tile x lists exactly the
    tiles holding an allowed pair against it, ascending, FULL exactly where the oracle's class is
    FULL; the kernels' bit-mask predicate over the listed tiles counts every row's allowed pairs
    exactly once."""
    lst, off = tsa.attn_bwd_lg_lists_host(S, w, G)
    n = (S + T - 1) // T
    assert off.shape == (n + 1,) and off[0] == 0 and off[-1] == lst.size
    classes = oracle.tile_classes(tsa.MASK_LOCAL_GLOBAL, S, w, list(G))  # [query tile, key tile]
    assert np.array_equal(classes, classes.T)  # the mask is symmetric
    for x in range(n):
        ent = [int(e) for e in lst[off[x]:off[x + 1]]]
        tiles = [e & (tsa.LIST_FULL - 1) for e in ent]
        assert tiles == sorted(set(tiles))
        assert tiles == [t for t in range(n) if classes[x, t] != 0], x
        for e, t in zip(ent, tiles):
            assert bool(e & tsa.LIST_FULL) == (classes[x, t] == 1), (x, t)
    counts = _lg_bwd_kernel_counts(S, w, G, lst, off)
    assert np.array_equal(counts, oracle.row_counts(tsa.MASK_LOCAL_GLOBAL, S, w, list(G)))


def test_lg_backward_lists_of_the_local_global_workload():
    """The 8K local + global workload (w 512, globals 0, 1000, 3000, 6000): tile classes against
    the oracle's enumeration; a tile holding a global lists every tile."""
    w = wl.LONGFORMER_8K
    lst, off = tsa.attn_bwd_lg_lists_host(w.S, w.window, w.globals_idx)
    classes = oracle.tile_classes(tsa.MASK_LOCAL_GLOBAL, w.S, w.window, list(w.globals_idx))
    n = w.S // T
    gt = {g // T for g in w.globals_idx}
    for x in range(n):
        ent = [int(e) for e in lst[off[x]:off[x + 1]]]
        assert [e & (tsa.LIST_FULL - 1) for e in ent] == [t for t in range(n) if classes[x, t] != 0]
        assert [bool(e & tsa.LIST_FULL) for e in ent] == [classes[x, t] == 1 for t in range(n) if classes[x, t]]
        if x in gt:
            assert len(ent) == n


def test_lg_backward_lists_reject_bad_arguments():
    for S, w, G in ((0, 1, ()), (100, -1, ()), (100, 3, (100,)), (100, 3, (-1,))):
        with pytest.raises(tsa.AttnError) as e:
            tsa.attn_bwd_lg_lists_host(S, w, G)
        assert e.value.status == tsa.ATTN_ERR_INVALID_ARG


def test_kv_schedule_rejects_local_global():
    with pytest.raises(tsa.AttnError) as e:
        tsa.attn_kv_schedule_host(300, tsa.MASK_LOCAL_GLOBAL, 5)
    assert e.value.status == tsa.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,Hq,Hkv,S,d,kind,w", [(2, 32, 32, 4096, 128, tsa.MASK_CAUSAL, 0),
                                                (1, 32, 8, 16384, 128, tsa.MASK_CAUSAL_SLIDING, 4095),
                                                (1, 64, 8, 32768, 128, tsa.MASK_CAUSAL, 0),
                                                (3, 6, 2, 300, 64, tsa.MASK_SLIDING, 40),
                                                (2, 4, 1, 129, 128, tsa.MASK_FULL, 0)])
def test_bwd_dq_order_is_a_grouped_permutation(B, Hq, Hkv, S, d, kind, w):
    """The dQ launch runs the forward's first-launch items, each once, grouped by kv head so that
    about 32 MB of K and V is live at a time, and in the forward's order within a group."""
    fwd, n_first = tsa.attn_schedule_host(B, Hq, Hkv, S, kind, w)
    fwd = fwd[:n_first]
    dq = tsa.attn_bwd_dq_schedule_host(B, Hq, Hkv, S, d, kind, w)
    assert sorted(map(tuple, dq.tolist())) == sorted(map(tuple, fwd.tolist()))
    kv_group = max(1, (32 << 20) // (4 * S * d))
    key = lambda it: ((it[0] // Hq) * Hkv + (it[0] % Hq) // (Hq // Hkv)) // kv_group
    keys = [key(it) for it in dq.tolist()]
    assert keys == sorted(keys)
    for k in set(keys):
        assert [it for it in dq.tolist() if key(it) == k] == [it for it in fwd.tolist() if key(it) == k]
