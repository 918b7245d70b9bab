// Host-side tile schedule builder (see schedule.h).
#include "schedule.h"

#include <algorithm>
#include <cmath>
#include <cstdint>

namespace attn {
namespace {

constexpr int T = ATTN_TILE;

// Allowed key interval [lo(i), hi(i)] of row i for the window part of a mask
// (global rows / columns are handled separately).  Both ends are
// non-decreasing in i for every kind, which the tile classification uses.
struct RowBand {
    int kind, S, w;
    long lo(long i) const {
        switch (kind) {
        case ATTN_MASK_SLIDING:
        case ATTN_MASK_LOCAL_GLOBAL:
        case ATTN_MASK_CAUSAL_SLIDING: return std::max(0L, i - w);
        default: return 0;
        }
    }
    long hi(long i) const {
        switch (kind) {
        case ATTN_MASK_CAUSAL:
        case ATTN_MASK_CAUSAL_SLIDING: return std::min<long>(i, S - 1);
        case ATTN_MASK_SLIDING:
        case ATTN_MASK_LOCAL_GLOBAL: return std::min<long>(S - 1, i + w);
        default: return S - 1;
        }
    }
};

}  // namespace

attn_status build_schedule(const ScheduleInput& in, Schedule* out) {
    const int S = in.S;
    const int nq = (S + T - 1) / T, nk = (S + T - 1) / T;
    const bool lg = in.kind == ATTN_MASK_LOCAL_GLOBAL;
    const int nG = lg ? (int)in.globals.size() : 0;
    RowBand band{in.kind, S, in.window};

    // prefix count of global positions: cntG[x] = #globals < x
    std::vector<int> is_g(S, 0), cntG(S + 1, 0);
    for (int g : in.globals) is_g[g] = 1;
    for (int x = 0; x < S; ++x) cntG[x + 1] = cntG[x] + is_g[x];
    auto globals_in = [&](long a, long b) -> long {  // #globals in [a, b]
        if (b < a) return 0;
        return cntG[b + 1] - cntG[a];
    };

    struct Proto { int q_tile, kv_begin, kv_end, full_begin, full_end, flags, n_gtiles; };
    std::vector<Proto> protos;
    protos.reserve(nq);
    const int n_gtiles = (nG + T - 1) / T;

    for (int qt = 0; qt < nq; ++qt) {
        const long r0 = (long)qt * T;
        const long r1 = std::min<long>(S, r0 + T) - 1;
        const bool rows_full = (r0 + T - 1) < S;
        const int kv_begin = (int)(band.lo(r0) / T);
        const int kv_end = (int)(band.hi(r1) / T) + 1;
        int full_begin = -1, full_end = -1;
        for (int t = kv_begin; t < kv_end; ++t) {
            const long c0 = (long)t * T, c1 = c0 + T - 1;
            const long c1s = std::min<long>(c1, S - 1);
            // at least one allowed pair: some row's interval meets [c0, c1s]
            bool any = false;
            for (long i = r0; i <= r1 && !any; ++i)
                any = band.lo(i) <= c1s && band.hi(i) >= c0;
            if (!any) return ATTN_ERR_UNSUPPORTED;  // interval masks never leave holes
            bool full = rows_full && c1 < S;
            if (full) {
                if (!lg) {
                    full = band.lo(r0 + T - 1) <= c0 && band.hi(r0) >= c1;
                } else {
                    for (long i = r0; i <= r0 + T - 1 && full; ++i) {
                        if (is_g[i]) continue;
                        const long lo = band.lo(i), hi = band.hi(i);
                        // columns of [c0, c1] outside [lo, hi] must all be global
                        const long a1 = c0, b1 = std::min(c1, lo - 1);
                        const long a2 = std::max(c0, hi + 1), b2 = c1;
                        long need = 0, have = 0;
                        if (b1 >= a1) { need += b1 - a1 + 1; have += globals_in(a1, b1); }
                        if (b2 >= a2) { need += b2 - a2 + 1; have += globals_in(a2, b2); }
                        full = need == have;
                    }
                }
            }
            if (full) {
                if (full_begin < 0) { full_begin = t; full_end = t + 1; }
                else if (full_end == t) full_end = t + 1;
                else return ATTN_ERR_UNSUPPORTED;  // FULL tiles must be contiguous
            }
        }
        if (full_begin < 0) full_begin = full_end = kv_begin;
        int flags = 0, ngt = 0;
        if (lg && nG > 0) {
            const long band_lo = (long)kv_begin * T, band_hi = (long)kv_end * T;  // [lo, hi)
            const long outside = nG - globals_in(band_lo, std::min<long>(band_hi, S) - 1);
            if (outside > 0) { flags |= ATTN_WORK_GLOBAL_COLS; ngt = (int)((outside + T - 1) / T); }
            if (globals_in(r0, r1) > 0) flags |= ATTN_WORK_HAS_GLOBAL_ROWS;
        }
        protos.push_back({qt, kv_begin, kv_end, full_begin, full_end, flags, ngt});
    }

    // longest first; equal cost -> later query tile first, then head order so
    // that the query heads of one key/value group run side by side
    std::vector<int> order(protos.size());
    for (size_t k = 0; k < order.size(); ++k) order[k] = (int)k;
    auto cost = [&](const Proto& p) { return (p.kv_end - p.kv_begin) + p.n_gtiles; };
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
        const int cx = cost(protos[x]), cy = cost(protos[y]);
        if (cx != cy) return cx > cy;
        return protos[x].q_tile > protos[y].q_tile;
    });

    // Long problems: the (batch, kv head) units are taken in groups whose K and V fit in about
    // 32 MB of L2 (at d = 128, the larger head size), every item of a group, longest first,
    // before the next group.  The query tiles that read the same K/V tiles then run together
    // and the K/V tiles come from DRAM about once.  Grouping delays the long items of the later
    // groups, which costs at the end of the launch; it is used only when every group holds at
    // least kMinGroupItems items (many waves of CTAs), so that this tail is small next to the
    // whole.  Otherwise one group: longest first over all heads.
    constexpr long kMinGroupItems = 4096;
    const int BH = in.B * in.Hq;
    const int group = in.Hq / in.Hkv;
    const long kv_bytes = 512L * S;  // K and V of one kv head: 2 * S * 128 * 2 bytes
    int g_kv = (int)std::max(1L, std::min((long)in.B * in.Hkv, (32L << 20) / kv_bytes));
    if ((long)g_kv * group * nq < kMinGroupItems) g_kv = in.B * in.Hkv;
    const int n_groups = (in.B * in.Hkv + g_kv - 1) / g_kv;
    out->items.clear();
    out->items.reserve((size_t)(protos.size() + (size_t)n_gtiles) * BH * ATTN_WORK_INTS);
    for (int gi = 0; gi < n_groups; ++gi) {
        const int u0 = gi * g_kv, u1 = std::min(in.B * in.Hkv, u0 + g_kv);  // kv units [u0, u1)
        for (int k : order) {
            const Proto& p = protos[k];
            for (int u = u0; u < u1; ++u) {
                const int b = u / in.Hkv, g = u % in.Hkv;
                for (int a = g * group; a < (g + 1) * group; ++a) {
                    const int it[ATTN_WORK_INTS] = {b * in.Hq + a, p.q_tile, p.kv_begin, p.kv_end,
                                                    p.full_begin, p.full_end, p.flags, p.n_gtiles};
                    out->items.insert(out->items.end(), it, it + ATTN_WORK_INTS);
                }
            }
        }
    }
    out->n_main = (int)protos.size() * BH;

    // dense pass for the global rows: every key, FULL except a ragged last tile.
    // The key tiles are split into chunks of about half the longest query-tile item (one
    // work item each).  They come after the band items, longest first, and fill the last,
    // partly empty wave of the launch instead of lengthening it; each chunk writes a partial
    // result and the last to finish merges them.
    out->n_grows = 0;
    out->n_chunks = 1;
    if (lg && nG > 0) {
        const int full_end = (S % T == 0) ? nk : nk - 1;
        int longest = 1;
        for (const Proto& p : protos) longest = std::max(longest, cost(p));
        const int per = std::max(1, std::min(nk, (longest + 1) / 2));
        const int chunks = (nk + per - 1) / per;  // no empty chunk
        out->n_chunks = chunks;
        for (int c = 0; c < chunks; ++c)
            for (int gt = 0; gt < n_gtiles; ++gt)
                for (int bh = 0; bh < BH; ++bh) {
                    const int kb = c * per, ke = std::min(nk, kb + per);
                    const int fe = std::max(kb, std::min(ke, full_end));  // FULL tiles [kb, fe)
                    const int it[ATTN_WORK_INTS] = {bh, gt, kb, ke, kb, fe, ATTN_WORK_GLOBAL_ROWS, c};
                    out->items.insert(out->items.end(), it, it + ATTN_WORK_INTS);
                    ++out->n_grows;
                }
    }
    out->gsplit.assign((size_t)nq * 2, 0);
    for (const Proto& p : protos) {  // #globals before the band, and #globals before its end
        const long band_lo = std::min<long>((long)p.kv_begin * T, S), band_hi = std::min<long>((long)p.kv_end * T, S);
        out->gsplit[(size_t)p.q_tile * 2] = cntG[band_lo];
        out->gsplit[(size_t)p.q_tile * 2 + 1] = cntG[band_hi];
    }
    out->n_kv_tiles = nk;
    out->n_global_tiles = n_gtiles;
    out->global_bits.assign((size_t)nk * 4, 0u);
    for (int g : in.globals) out->global_bits[(size_t)(g / T) * 4 + (g % T) / 32] |= 1u << (g % 32);
    return ATTN_OK;
}

attn_status build_kv_schedule(int S, int kind, int window, std::vector<int>* items) {
    if (kind == ATTN_MASK_LOCAL_GLOBAL) return ATTN_ERR_UNSUPPORTED;
    const long w = window;
    // rows i that see key j form [ilo(j), ihi(j)]; both ends are non-decreasing in j
    auto ilo = [&](long j) -> long {
        switch (kind) {
        case ATTN_MASK_CAUSAL:
        case ATTN_MASK_CAUSAL_SLIDING: return j;
        case ATTN_MASK_SLIDING: return std::max(0L, j - w);
        default: return 0;
        }
    };
    auto ihi = [&](long j) -> long {
        switch (kind) {
        case ATTN_MASK_CAUSAL_SLIDING:
        case ATTN_MASK_SLIDING: return std::min<long>(S - 1, j + w);
        default: return S - 1;
        }
    };
    const int nk = (S + T - 1) / T;
    struct Item { int kt, qb, qe, fb, fe; };
    std::vector<Item> v;
    for (int kt = 0; kt < nk; ++kt) {
        const long j0 = (long)kt * T, j1 = std::min<long>(S, j0 + T) - 1;
        const int qb = (int)(ilo(j0) / T), qe = (int)(ihi(j1) / T) + 1;
        const bool keys_full = j0 + T - 1 < S;
        int fb = -1, fe = -1;
        for (int qt = qb; qt < qe; ++qt) {
            const long r0 = (long)qt * T;
            const bool full = keys_full && r0 + T - 1 < S && r0 >= ilo(j1) && r0 + T - 1 <= ihi(j0);
            if (full) {
                if (fb < 0) { fb = qt; fe = qt + 1; }
                else if (fe == qt) fe = qt + 1;
                else return ATTN_ERR_UNSUPPORTED;  // cannot happen for interval masks
            }
        }
        if (fb < 0) fb = fe = qb;
        v.push_back({kt, qb, qe, fb, fe});
    }
    std::stable_sort(v.begin(), v.end(), [](const Item& x, const Item& y) {
        if (x.qe - x.qb != y.qe - y.qb) return x.qe - x.qb > y.qe - y.qb;
        return x.kt < y.kt;
    });
    items->clear();
    for (const Item& it : v) {
        const int a[ATTN_WORK_INTS] = {it.kt, it.qb, it.qe, it.fb, it.fe, 0, 0, 0};
        items->insert(items->end(), a, a + ATTN_WORK_INTS);
    }
    return ATTN_OK;
}

int dq_kv_group(int S, int d_k) {
    const long per_head = 2L * S * d_k * 2;  // K and V of one kv head, bf16
    return (int)std::max(1L, std::min(1L << 20, (32L << 20) / std::max(1L, per_head)));
}

std::vector<int> order_dq_items(const std::vector<int>& items, int n_items, int Hq, int Hkv, int kv_group) {
    const int group = Hq / Hkv;
    auto key = [&](int k) {
        const int bh = items[(size_t)k * ATTN_WORK_INTS];
        return ((bh / Hq) * Hkv + (bh % Hq) / group) / kv_group;
    };
    std::vector<int> order(n_items);
    for (int k = 0; k < n_items; ++k) order[k] = k;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return key(x) < key(y); });
    std::vector<int> out;
    out.reserve((size_t)n_items * ATTN_WORK_INTS);
    for (int k : order) out.insert(out.end(), items.begin() + (size_t)k * ATTN_WORK_INTS,
                                   items.begin() + (size_t)(k + 1) * ATTN_WORK_INTS);
    return out;
}

void build_lg_pair_lists(int S, int window, const std::vector<int>& globals, std::vector<int>* list,
                         std::vector<int>* offsets) {
    const int n = (S + T - 1) / T;
    RowBand band{ATTN_MASK_LOCAL_GLOBAL, S, window};
    std::vector<int> is_g(S, 0), cntG(S + 1, 0);
    for (int g : globals) is_g[g] = 1;
    for (int x = 0; x < S; ++x) cntG[x + 1] = cntG[x] + is_g[x];
    auto globals_in = [&](long a, long b) -> long { return b < a ? 0 : cntG[b + 1] - cntG[a]; };
    list->clear();
    offsets->assign((size_t)n + 1, 0);
    for (int x = 0; x < n; ++x) {
        const long r0 = (long)x * T, r1 = std::min<long>(S, r0 + T) - 1;
        const bool x_has_g = globals_in(r0, r1) > 0;
        const int band_lo = (int)(band.lo(r0) / T), band_hi = (int)(band.hi(r1) / T);  // inclusive
        const bool x_all_g = r0 + T - 1 < S && globals_in(r0, r0 + T - 1) == T;
        for (int t = 0; t < n; ++t) {
            const long c0 = (long)t * T, c1 = c0 + T - 1, c1s = std::min<long>(c1, S - 1);
            const bool t_has_g = globals_in(c0, c1s) > 0;
            const bool in_band = t >= band_lo && t <= band_hi;
            if (!x_has_g && !t_has_g && !in_band) continue;
            // every pair allowed: both tiles whole, and each row global or its window plus the
            // global columns covering [c0, c1].  Outside the band no row's window reaches the tile
            // (the band is the union of the rows' windows), so only a tile of global rows or of
            // global columns is FULL there: an O(1) test instead of the per-row one.
            bool full = r0 + T - 1 < S && c1 < S;
            if (full && !in_band) {
                list->push_back(t | ((x_all_g || globals_in(c0, c1) == T) ? ATTN_LIST_FULL : 0));
                continue;
            }
            for (long i = r0; i <= r0 + T - 1 && full; ++i) {
                if (is_g[i]) continue;
                const long lo = band.lo(i), hi = band.hi(i);
                const long a1 = c0, b1 = std::min(c1, lo - 1), a2 = std::max(c0, hi + 1), b2 = c1;
                long need = 0, have = 0;
                if (b1 >= a1) { need += b1 - a1 + 1; have += globals_in(a1, b1); }
                if (b2 >= a2) { need += b2 - a2 + 1; have += globals_in(a2, b2); }
                full = need == have;
            }
            list->push_back(t | (full ? ATTN_LIST_FULL : 0));
        }
        (*offsets)[(size_t)x + 1] = (int)list->size();
    }
}

void build_lg_bwd_items(int B, int Hq, int Hkv, int S, int d_k, const std::vector<int>& offsets, std::vector<int>* dq_items,
                        std::vector<int>* kv_items) {
    const int n = (int)offsets.size() - 1;
    std::vector<int> order(n);
    for (int x = 0; x < n; ++x) order[x] = x;
    // longest first; equal length -> tile order
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
        return offsets[x + 1] - offsets[x] > offsets[y + 1] - offsets[y];
    });
    kv_items->clear();
    for (int x : order) {
        const int it[ATTN_WORK_INTS] = {x, offsets[x], offsets[x + 1], 0, 0, 0, 0, 0};
        kv_items->insert(kv_items->end(), it, it + ATTN_WORK_INTS);
    }
    std::vector<int> q;
    q.reserve((size_t)n * B * Hq * ATTN_WORK_INTS);
    for (int x : order)
        for (int bh = 0; bh < B * Hq; ++bh) {
            const int it[ATTN_WORK_INTS] = {bh, x, offsets[x], offsets[x + 1], 0, 0, 0, 0};
            q.insert(q.end(), it, it + ATTN_WORK_INTS);
        }
    *dq_items = order_dq_items(q, n * B * Hq, Hq, Hkv, dq_kv_group(S, d_k));
}

void decode_tile_range(int kind, int S_q, int window, int L, int* lo, int* hi) {
    *lo = kind == ATTN_MASK_CAUSAL_SLIDING ? std::max(0, L - S_q - window) / T : 0;
    *hi = (L + T - 1) / T;
}

void build_decode_schedule(int B, int Hkv, int S_q, int kind, int window, const int* lens, int n_sm,
                           DecodeSchedule* out) {
    out->tile_prefix.assign(B + 1, 0);
    for (int b = 0; b < B; ++b) {
        int lo, hi;
        decode_tile_range(kind, S_q, window, lens[b], &lo, &hi);
        out->tile_prefix[b + 1] = out->tile_prefix[b] + (hi - lo);
    }
    out->total_tiles = (long long)Hkv * out->tile_prefix[B];
    out->n_cta = (int)std::min<long long>(std::max(1, n_sm), out->total_tiles);
    // Share boundaries at equal steps of F(i) = i + a * (unit begins in (0, i]): within unit j
    // (indices [ub[j], ub[j+1])) F(i) = i + a * j, so the weight of a share is its tiles plus a
    // for every unit begun inside it.  Every share keeps at least one tile.
    const int n = out->n_cta;
    const long long T = out->total_tiles;
    const double a = kDecodeStretchCost;
    std::vector<long long> ub;  // unit begins in list order; ub[0] = 0
    ub.reserve((size_t)B * Hkv + 1);
    for (int b = 0; b < B; ++b) {
        const int n_b = out->tile_prefix[b + 1] - out->tile_prefix[b];
        for (int g = 0; g < Hkv && n_b > 0; ++g) ub.push_back((long long)Hkv * out->tile_prefix[b] + (long long)g * n_b);
    }
    ub.push_back(T);  // sentinel
    const double F_T = (double)T + a * (double)(ub.size() - 2);
    out->share.assign(n + 1, 0);
    out->share[n] = T;
    size_t j = 0;
    for (int k = 1; k < n; ++k) {
        const double tau = F_T * k / n;
        while (j + 2 < ub.size() && (double)(ub[j + 1] - 1) + a * (double)j < tau) ++j;
        long long i = std::max(ub[j], (long long)std::ceil(tau - a * (double)j));
        i = std::max(i, out->share[k - 1] + 1);
        i = std::min(i, T - (n - k));
        out->share[k] = i;
    }
}

}  // namespace attn
