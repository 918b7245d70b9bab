"""The decode work split (host only) against brute force from the oracle's decode predicate.

The kernel's arithmetic is restated here: unit (b, g) covers the indices
[Hkv * prefix[b] + g * n_b, ... + n_b) of one list of T tiles, and CTA k takes
[share[k], share[k+1]).  Checked bit-exactly, without a GPU:
  * every key tile a sequence needs (some query row may see one of its keys, by
    enumeration of the oracle's predicate) is in its range, and the range starts
    and ends at such tiles;
  * every tile of every unit belongs to exactly one CTA; the shares are contiguous
    and non-empty, and their boundaries sit at equal steps of the weight
    F(i) = i + 2 * (unit begins in (0, i]) (tiles plus two per extra stretch);
  * only a CTA's first and last stretches can be partial units, and the partial-
    result slots the writers use (2k for a first stretch, 2k+1 for a last one)
    are exactly the slots the merge of each unit enumerates.
"""
import bisect
import random

import pytest

import oracle
import transformer_self_attention_gb300 as tsa

T = tsa.TILE
KINDS = (tsa.MASK_FULL, tsa.MASK_CAUSAL, tsa.MASK_CAUSAL_SLIDING)


def _tile_lo(kind, S_q, window, L):
    return max(0, L - S_q - window) // T if kind == tsa.MASK_CAUSAL_SLIDING else 0


def _needed_tiles(kind, S_q, window, L):
    tiles = set()
    for i in range(S_q):
        t = L - S_q + i
        for j in range(L):
            if oracle.decode_allowed(kind, t, j, L, window):
                tiles.add(j // T)
    return tiles


STRETCH_COST = 2


def _stretches(Hkv, prefix, share, k):
    """The kernel's walk over CTA k's share: list of (b, g, first_tile_in_unit, count, whole)."""
    i, end = int(share[k]), int(share[k + 1])
    out = []
    while i < end:
        b = max(x for x in range(len(prefix) - 1) if Hkv * prefix[x] <= i)
        n_b = prefix[b + 1] - prefix[b]
        r = i - Hkv * prefix[b]
        g, t_in = r // n_b, r % n_b
        unit_begin = Hkv * prefix[b] + g * n_b
        count = min(end, unit_begin + n_b) - i
        out.append((b, g, t_in, count, t_in == 0 and count == n_b))
        i += count
    return out


def _share_of(i, share):
    """The CTA whose share holds index i (the last one beginning at or before i)."""
    return max(k for k in range(len(share) - 1) if share[k] <= i)


def _unit_begins(Hkv, prefix):
    return [Hkv * prefix[b] + g * (prefix[b + 1] - prefix[b]) for b in range(len(prefix) - 1) for g in range(Hkv)]


def _weight(i, begins):
    """F(i): tiles before i plus the stretch cost of every unit begun in (0, i]."""
    pos = sorted(u for u in begins if u > 0)
    return i + STRETCH_COST * bisect.bisect_right(pos, i)


def _check_shares(share, n_cta, total, begins):
    share = [int(x) for x in share]
    assert len(share) == n_cta + 1 and share[0] == 0 and share[-1] == total
    assert all(share[k] < share[k + 1] for k in range(n_cta)), "an empty share"
    F_T = total + STRETCH_COST * (len(begins) - 1)
    pos = sorted(u for u in begins if u > 0)
    F = lambda i: i + STRETCH_COST * bisect.bisect_right(pos, i)  # non-decreasing in i
    for k in range(1, n_cta):
        tau = F_T * k / n_cta
        lo, hi = share[k - 1] + 1, total - (n_cta - k)  # room for one tile per remaining CTA
        a, b = 0, total  # smallest i with F(i) >= tau, by bisection (F(total) >= tau)
        while a < b:
            mid = (a + b) // 2
            if F(mid) >= tau - 1e-9:
                b = mid
            else:
                a = mid + 1
        assert share[k] == min(max(a, lo), hi), (k, share[k], a, lo, hi)


def _check(B, Hkv, S_q, S_cap, kind, window, lens, n_sm):
    n_cta, prefix, share = tsa.attn_decode_schedule_host(B, Hkv, S_q, S_cap, kind, window, lens, n_sm)
    prefix = [int(x) for x in prefix]
    total = Hkv * prefix[B]
    assert n_cta == min(n_sm, 512, total)
    _check_shares(share, n_cta, total, _unit_begins(Hkv, prefix))
    # ranges of the sequences
    for b, L in enumerate(lens):
        lo = _tile_lo(kind, S_q, window, L)
        hi = (L + T - 1) // T
        assert prefix[b + 1] - prefix[b] == hi - lo
        need = _needed_tiles(kind, S_q, window, L)
        assert need <= set(range(lo, hi)) and min(need) == lo and max(need) == hi - 1
    # cover, balance, partial stretches and their slots
    seen = {}
    writer_slots = {}
    sizes = []
    for k in range(n_cta):
        st = _stretches(Hkv, prefix, share, k)
        sizes.append(sum(c for _, _, _, c, _ in st))
        for idx, (b, g, t_in, count, whole) in enumerate(st):
            for t in range(t_in, t_in + count):
                assert (b, g, t) not in seen
                seen[(b, g, t)] = k
            if not whole:
                assert idx == 0 or idx == len(st) - 1, "a partial stretch in the middle of a share"
                writer_slots.setdefault((b, g), set()).add(2 * k + (0 if idx == 0 else 1))
    assert len(seen) == total
    for (b, g), slots in writer_slots.items():
        n_b = prefix[b + 1] - prefix[b]
        unit_begin = Hkv * prefix[b] + g * n_b
        k0, k1 = _share_of(unit_begin, share), _share_of(unit_begin + n_b - 1, share)
        k0_first = share[k0] == unit_begin
        merge = {2 * k0 + (0 if k0_first else 1)} | {2 * kk for kk in range(k0 + 1, k1 + 1)}
        assert slots == merge, (b, g, slots, merge)
        assert len(slots) == k1 - k0 + 1 >= 2
    return n_cta, prefix


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("S_q", [1, 2, 5])
def test_decode_split_covers_the_allowed_keys(kind, S_q):
    rng = random.Random(kind * 10 + S_q)
    for trial in range(6):
        B = rng.randint(1, 5)
        Hkv = rng.choice([1, 2, 8])
        S_cap = max(rng.choice([S_q, 127, 128, 129, 300, 1000]), S_q)
        lens = [rng.randint(S_q if kind != tsa.MASK_FULL else 1, S_cap) for _ in range(B)]
        window = rng.choice([0, 1, 127, 128, 200])
        _check(B, Hkv, S_q, S_cap, kind, window, lens, n_sm=rng.choice([1, 3, 7, 152]))


def test_decode_split_long_ragged_batch():
    """Eight ragged 16K..30K caches with 8 kv heads on 152 SMs: units cut across CTAs, and the
    shares' weights (tiles plus the cost of every extra stretch) equal to within one stretch."""
    lens = [16384 + 2000 * b for b in range(8)]
    n_cta, prefix, share = tsa.attn_decode_schedule_host(8, 8, 1, 32768, tsa.MASK_CAUSAL, 0, lens, 152)
    prefix = [int(x) for x in prefix]
    total = 8 * prefix[-1]
    assert n_cta == 152
    begins = _unit_begins(8, prefix)
    _check_shares(share, n_cta, total, begins)
    cost = [int(share[k + 1] - share[k]) + STRETCH_COST * sum(1 for u in begins if share[k] < u < share[k + 1])
            for k in range(n_cta)]
    assert max(cost) - min(cost) <= 1 + STRETCH_COST
    # a share holding an extra stretch is shorter than one that does not
    two = [int(share[k + 1] - share[k]) for k in range(n_cta) if any(share[k] < u < share[k + 1] for u in begins)]
    one = [int(share[k + 1] - share[k]) for k in range(n_cta) if not any(share[k] < u < share[k + 1] for u in begins)]
    assert two and one and max(two) < min(one) + 1


def test_decode_split_single_huge_unit():
    """One long sequence with one kv head is spread over every CTA."""
    n_cta, prefix, share = tsa.attn_decode_schedule_host(1, 1, 1, 1 << 20, tsa.MASK_CAUSAL, 0, [1 << 20], 152)
    assert n_cta == 152 and prefix[1] == (1 << 20) // T
    sizes = [int(share[k + 1] - share[k]) for k in range(n_cta)]
    assert max(sizes) - min(sizes) <= 1  # one unit: no stretch to weigh


def test_decode_split_fewer_tiles_than_sms():
    n_cta, prefix, share = tsa.attn_decode_schedule_host(2, 1, 1, 300, tsa.MASK_CAUSAL, 0, [1, 200], 152)
    assert n_cta == 3 and list(prefix) == [0, 1, 3] and list(share) == [0, 1, 2, 3]


def test_decode_sliding_window_skips_old_tiles():
    """The causal window reads only the tiles of the last window + S_q positions."""
    L, w = 16384, 4095
    n_cta, prefix, share = tsa.attn_decode_schedule_host(1, 8, 1, L, tsa.MASK_CAUSAL_SLIDING, w, [L], 152)
    assert prefix[1] == L // T - (L - 1 - w) // T


@pytest.mark.parametrize("args,status", [
    ((1, 1, 1, 8, tsa.MASK_SLIDING, 2, [8], 4), tsa.ATTN_ERR_UNSUPPORTED),       # not a decode kind
    ((1, 1, 1, 8, tsa.MASK_LOCAL_GLOBAL, 2, [8], 4), tsa.ATTN_ERR_UNSUPPORTED),
    ((1, 1, 65, 100, tsa.MASK_CAUSAL, 0, [100], 4), tsa.ATTN_ERR_UNSUPPORTED),   # more than 64 rows
    ((1, 1, 4, 8, tsa.MASK_CAUSAL, 0, [3], 4), tsa.ATTN_ERR_INVALID_ARG),        # fewer cached than new rows
    ((1, 1, 1, 8, tsa.MASK_CAUSAL, 0, [9], 4), tsa.ATTN_ERR_INVALID_ARG),        # beyond the capacity
    ((1, 1, 1, 8, tsa.MASK_CAUSAL, 0, [0], 4), tsa.ATTN_ERR_INVALID_ARG),        # empty cache
    ((1, 1, 1, 8, tsa.MASK_CAUSAL_SLIDING, -1, [8], 4), tsa.ATTN_ERR_INVALID_ARG),
    ((1, 1, 1, 8, tsa.MASK_CAUSAL, 0, [8], 0), tsa.ATTN_ERR_INVALID_ARG),        # no multiprocessor
    ((1025, 1, 1, 8, tsa.MASK_CAUSAL, 0, [8] * 1025, 4), tsa.ATTN_ERR_UNSUPPORTED),
])
def test_decode_schedule_validation(args, status):
    with pytest.raises(tsa.AttnError) as e:
        tsa.attn_decode_schedule_host(*args)
    assert e.value.status == status


def test_cross_attention_lengths_may_be_shorter_than_the_query_rows():
    n_cta, prefix, share = tsa.attn_decode_schedule_host(2, 4, 32, 4096, tsa.MASK_FULL, 0, [3, 4096], 152)
    assert list(prefix) == [0, 1, 33]


@pytest.mark.parametrize("kw,status", [
    (dict(B=1, Hq=4, Hkv=4, S_q=1, S_cap=64, d_k=96, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_UNSUPPORTED),
    (dict(B=1, Hq=4, Hkv=4, S_q=1, S_cap=64, d_k=64, scale=0.0, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_INVALID_ARG),
    (dict(B=1, Hq=4, Hkv=3, S_q=1, S_cap=64, d_k=64, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_INVALID_ARG),
    (dict(B=1, Hq=64, Hkv=1, S_q=2, S_cap=64, d_k=64, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_UNSUPPORTED),
    (dict(B=1, Hq=4, Hkv=4, S_q=8, S_cap=4, d_k=64, scale=0.1, kind=tsa.MASK_CAUSAL), tsa.ATTN_ERR_INVALID_ARG),
    (dict(B=1, Hq=4, Hkv=4, S_q=1, S_cap=64, d_k=64, scale=0.1, kind=tsa.MASK_SLIDING), tsa.ATTN_ERR_UNSUPPORTED),
])
def test_decode_create_rejects_bad_arguments_before_any_cuda_call(kw, status):
    with pytest.raises(tsa.AttnError) as e:
        tsa.attn_decode_create(**kw)
    assert e.value.status == status


def test_decode_split_grid_capped_at_512_ctas():
    """More multiprocessors than the parameter table holds: the grid stops at 512 CTAs, and the
    shares still cover the list with the weighted boundaries."""
    lens = [4096] * 64
    n_cta, prefix, share = tsa.attn_decode_schedule_host(64, 8, 1, 4096, tsa.MASK_CAUSAL, 0, lens, 700)
    prefix = [int(x) for x in prefix]
    total = 8 * prefix[-1]
    assert n_cta == 512 and len(share) == 513
    _check_shares(share, n_cta, total, _unit_begins(8, prefix))


def test_decode_split_many_short_units():
    """Many two-tile units (ragged short caches): shares span several units, every tile is still
    covered once, partial units stay at the ends of a share, and the weights balance."""
    rng = random.Random(7)
    lens = [rng.randint(129, 256) for _ in range(96)]
    _check(96, 4, 1, 256, tsa.MASK_CAUSAL, 0, lens, 152)
    n_cta, prefix, share = tsa.attn_decode_schedule_host(96, 4, 1, 256, tsa.MASK_CAUSAL, 0, lens, 152)
    prefix = [int(x) for x in prefix]
    begins = _unit_begins(4, prefix)
    # each boundary sits within one step (a tile plus a unit begin) above its target of F, so two
    # shares' weights F(share[k + 1]) - F(share[k]) differ by less than two steps
    weight = [_weight(int(share[k + 1]), begins) - _weight(int(share[k]), begins) for k in range(n_cta)]
    assert max(weight) - min(weight) < 2 * (1 + STRETCH_COST)
