// Decode / key-value-cache attention for sm_103a (bf16 in, fp32 accumulation).
//
// What it computes: for each sequence b with cache_len[b] = L cached positions
// and S_q new query rows at positions L - S_q + i, every query head a attends
// to the cached keys and values of its kv head g(a) = a / (Hq / Hkv) under the
// mask kind (FULL for cross-attention, CAUSAL, CAUSAL_SLIDING).  This is the
// step-t output Softmax(q_t K_{1:t}^T / sqrt(d_k)) V_{1:t} of "Trasformer 浅析"
// (atffang.github.io), section 推理：KV 缓存, over the ragged batches and
// chunked prefill of "第 8 章 现代大模型架构" (theaiera.top), section
// 预填充创建缓存，解码复用缓存, and the n_dec x n_enc cross-attention of
// "Trasformer 浅析", section 交叉注意力.
//
// The work is bound by HBM: every key and value byte serves only the
// group * S_q query rows of its kv head.  So a CTA takes ALL query rows of one
// kv head's group at once (a GQA/MQA group reads its shared cache once,
// "第 8 章", 8.2.2 on MQA's single HBM read for h heads), and the tensor-core
// products are transposed so that the 128 keys of a tile fill the MMA's M
// dimension and the packed query rows its N dimension (NP = 16, 32 or 64):
//
//   S^T [128 keys x NP]  = K_tile [128 x d]  . Q^T [d x NP]      (both K-major)
//   O^T [d x NP]        += V_tile^T [d x 128] . P^T [128 x NP]   (V MN-major)
//
// Balance: the grid is persistent (one CTA per SM).  All (sequence, kv head)
// units are laid end to end as one list of key tiles and every CTA takes a
// contiguous share of it (the host weights a share by its tiles plus the cost
// of every unit begun inside it), so a CTA may finish the end of one unit and
// start the next.  A unit cut between CTAs yields partial results (O
// normalised by its own sum, and its LSE), combined with weights
// e^{LSE_c - LSE} by decode_merge_kernel, a programmatic dependent launch behind
// this kernel, or (merge mode 1) by the last CTA of the unit to finish (an
// arrival counter per unit that wraps back to zero).
//
//   warp 4 (producer) : TMA loads of each unit's packed Q rows (double-
//                       buffered) and of the K and V tiles into one ring of
//                       tile-sized 128B-swizzled slots (K of tile n, then V of
//                       tile n, in consecutive slots; K's slot is freed by its
//                       QK product, V's by its PV product, so as many slots as
//                       shared memory holds are in flight).
//   warp 5 (MMA)      : one thread issues QK(n+1) before PV(n) so that the
//                       softmax of tile n+1 overlaps the PV of tile n (S^T is
//                       double-buffered in tensor memory, P^T in shared memory).
//   warps 0-3         : thread t owns key t of the tile (tensor-memory lane t)
//                       and component t of d in O^T.  Running max m and sums
//                       in exp2 units of log2(e)-prescaled scores.  A tile
//                       first checks every allowed score against its row's
//                       running max; only when one exceeds it by more than 2^8
//                       (always on a unit's first tile) are the exact tile
//                       maxima formed (warp max reductions plus a 4-warp
//                       exchange) and O^T and the sums rescaled.  P^T goes to
//                       shared memory in the MMA's K-major swizzled layout.
//
// Stale cache entries (positions >= cache_len[b]) are never used: their scores
// are masked, and the V rows of a sequence's last tile past its length are
// zeroed in shared memory before the PV product (0 * NaN would be NaN).
// Every mbarrier wait is bounded by the watchdog limit; after a wait runs out
// the CTA records an error bit, drains its copies and MMAs and exits.
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

#include "device_once.h"
#include "kernels.h"
#include "sm103_ptx.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int BN = 128;         // keys per tile (the MMA's M)
constexpr int NTHREADS = 192;   // 4 softmax warps + producer + MMA
constexpr int WARP_PRODUCER = 4;
constexpr int WARP_MMA = 5;
constexpr int MAX_SLOTS = 12;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
constexpr int SMEM_LIMIT = 227 * 1024;   // one CTA per SM
constexpr int SMEM_HALF = 228 * 1024 / 2 - 1024;  // each of two CTAs per SM (1 KB reserved per CTA)

enum : int { ERR_PRODUCER = 1, ERR_MMA = 2, ERR_SOFTMAX = 4 };

template <int D, int NP>
struct DCfg {
    static constexpr int TB = BN * D * 2;         // one K or V tile
    static constexpr int SUB = BN * 128;          // one 64-column block of a K/V tile
    static constexpr int QT = NP * D * 2;         // one packed Q tile
    static constexpr int QB = NP * 128;           // one 64-column block of it
    static constexpr int PB = NP * 128;           // one 64-key half of a P^T buffer
    static constexpr int ZERO = (D == 64) ? SUB : 0;  // rows 64..127 of V^T when d = 64 (zeros)
    static constexpr int CTL = NP == 64 ? 8192 : 4096;  // DShared<NP>
    // At d = 64 with up to 32 packed rows the single MMA-issuing thread, not the memory, sets a
    // tile's pace (12 small products per 32 KB of K and V): two CTAs per SM, each with its own
    // issuing thread and half the shared memory.
    static constexpr int CTAS = (D == 64 && NP <= 32) ? 2 : 1;
    static constexpr int FIXED = 2 * QT + 2 * 2 * PB + ZERO + CTL + 1024;
    static constexpr int SLOTS_FIT = ((CTAS == 2 ? SMEM_HALF : SMEM_LIMIT) - FIXED) / TB;
    static constexpr int SLOTS = SLOTS_FIT > MAX_SLOTS ? MAX_SLOTS : SLOTS_FIT;  // K/V ring
    static_assert(SLOTS >= 4, "shared memory");
    static constexpr int OFF_KV = 0;
    static constexpr int OFF_Z = OFF_KV + SLOTS * TB;
    static constexpr int OFF_Q = OFF_Z + ZERO;
    static constexpr int OFF_P = OFF_Q + 2 * QT;
    static constexpr int OFF_CTL = OFF_P + 2 * 2 * PB;
    static constexpr int SMEM_ALLOC = OFF_CTL + CTL + 1024;
    static constexpr uint32_t TMEM_COLS = (3 * NP <= 64) ? 64 : (3 * NP <= 128) ? 128 : 256;
    static constexpr uint32_t TMEM_S = 0;       // S^T buffers: columns [0, NP) and [NP, 2 NP)
    static constexpr uint32_t TMEM_O = 2 * NP;  // O^T: columns [2 NP, 3 NP)
};

enum Bar {
    B_QFULL = 0,                      // 2: packed Q tile loaded
    B_QEMPTY = B_QFULL + 2,           // 2: last QK of its unit done (MMA commit)
    B_FULL = B_QEMPTY + 2,            // SLOTS: K/V slot loaded
    B_EMPTY = B_FULL + MAX_SLOTS,     // SLOTS: K/V slot read by its product (MMA commit)
    B_SFULL = B_EMPTY + MAX_SLOTS,    // 2: S^T buffer ready (MMA commit)
    B_PFULL = B_SFULL + 2,            // 2: P^T written, S^T read, O^T rescaled / read out (128 arrivals)
    B_PFREE = B_PFULL + 2,            // 2: PV(n) done, n of that parity (MMA commit)
    NBAR = B_PFREE + 2
};

template <int NP>
struct DShared {
    uint64_t bar[NBAR];
    alignas(16) float m[NP];   // running max of each packed row (log2 units)
    alignas(16) float alpha[NP];
    alignas(16) float inv_l[NP];
    alignas(16) float lse[NP];
    alignas(16) float bm[NP];  // ALiBi: slope of the row's head times log2(e)
    alignas(16) float bp[NP];  // ALiBi: the row's position t
    int lo[NP], hi[NP];        // allowed key interval of each packed row in the current unit
    int wmax[4][NP];           // per-warp tile maxima (order-preserving int encoding)
    float lsum[4][NP];
    uint32_t tmem_base;
    volatile int abort;
    int is_last;
    int flag;                  // a row of this tile needs O^T and the sums rescaled
};

struct Watch {
    volatile int* abort;
    int* err;
    long long ns;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Watch& w, int role) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 127u) == 0) {
            if (*w.abort) return false;
            if ((long long)(globaltimer() - t0) > w.ns) {
                *w.abort = 1;
                atomicOr(w.err, role);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Watch& w) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if ((long long)(globaltimer() - t0) > w.ns) return;
}

// float <-> int with the same order (for integer max reductions); -inf maps to the smallest value
__device__ __forceinline__ int ordered(float f) {
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float unordered(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

// 32 lanes x 16 columns of 32 bit into elements [OFF, OFF + 16) of a larger register array
template <int OFF, int N>
__device__ __forceinline__ void tmem_ld16_at(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(OFF + 16 <= N, "range");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]), "=r"(r[OFF + 4]),
          "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]), "=r"(r[OFF + 8]), "=r"(r[OFF + 9]),
          "=r"(r[OFF + 10]), "=r"(r[OFF + 11]), "=r"(r[OFF + 12]), "=r"(r[OFF + 13]), "=r"(r[OFF + 14]),
          "=r"(r[OFF + 15])
        : "r"(taddr));
}

// named barrier with an OR reduction of one predicate
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- the shared tile list
// First index of CTA k's share, and the CTA whose share holds index i.
// The shares are contiguous, non-empty and in CTA order (the host weights them by tiles and
// by the units begun inside them).
__device__ __forceinline__ long long share_begin(const DecodeParams& p, int k) { return p.share[k]; }
__device__ __forceinline__ int share_of(const DecodeParams& p, long long i) {
    int lo = 0, hi = p.n_cta - 1;  // the last CTA whose share begins at or before i
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.share[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// One unit's stretch of a CTA's share.
struct Seg {
    int b, g;
    int L;             // cache length of the sequence
    int n_unit;        // key tiles of the unit
    int tile0;         // first key tile (absolute) of this stretch
    int count;         // tiles in this stretch
    long long unit_begin;
    bool whole;        // the stretch is the whole unit
};

__device__ __forceinline__ Seg seg_at(const DecodeParams& p, long long i, long long end) {
    int lo = 0, hi = p.B - 1;  // last sequence whose first index is <= i
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)p.Hkv * p.tile_prefix[mid] <= i) lo = mid; else hi = mid - 1;
    }
    Seg s;
    s.b = lo;
    s.n_unit = p.tile_prefix[lo + 1] - p.tile_prefix[lo];
    const long long r = i - (long long)p.Hkv * p.tile_prefix[lo];
    s.g = (int)(r / s.n_unit);
    const int t_in = (int)(r - (long long)s.g * s.n_unit);
    s.unit_begin = (long long)p.Hkv * p.tile_prefix[lo] + (long long)s.g * s.n_unit;
    s.count = (int)(min(end, s.unit_begin + s.n_unit) - i);
    s.whole = t_in == 0 && s.count == s.n_unit;
    s.L = p.len[lo];
    const int t_lo = p.kind == ATTN_MASK_CAUSAL_SLIDING ? max(0, s.L - p.S_q - p.window) / BN : 0;
    s.tile0 = t_lo + t_in;
    return s;
}

// Position in a CTA's share: stretch j (its Seg s), tile q of it.
struct Walk {
    long long i;   // first index of the current stretch
    Seg s;
    int j, q;
    bool valid;
};
__device__ __forceinline__ Walk walk_begin(const DecodeParams& p, long long begin, long long end) {
    Walk w;
    w.i = begin;
    w.j = 0;
    w.q = 0;
    w.valid = begin < end;
    if (w.valid) w.s = seg_at(p, begin, end);
    return w;
}
__device__ __forceinline__ void walk_next(const DecodeParams& p, Walk& w, long long end) {
    if (!w.valid) return;
    if (++w.q < w.s.count) return;
    w.i += w.s.count;
    ++w.j;
    w.q = 0;
    w.valid = w.i < end;
    if (w.valid) w.s = seg_at(p, w.i, end);
}

// Partial-result slot of a stretch: 2k for the first stretch of CTA k's share, 2k+1 for its
// last (only these two can be partial).
__device__ __forceinline__ int part_slot(int k, bool first_of_share) { return 2 * k + (first_of_share ? 0 : 1); }

// Combine the partial results of unit (b, g) once all its stretches have arrived.  Warp w
// takes rows w, w+4, ...; every load of a phase is independent of the others, so the whole
// merge costs a few L2 round trips: (1) lane l reads LSE_c of partial c = l (+32, ...) for
// all the warp's rows, and warp reductions give M = max_c LSE_c and W = sum_c e^{LSE_c - M};
// (2) lane l accumulates d components [l*D/32, (l+1)*D/32) of sum_c e^{LSE_c - M} O_c / W,
// four partials and all rows at a time.  scratch_m / scratch_w: NP floats of shared memory.
template <int D, int NP>
__device__ void merge_unit(const DecodeParams& p, const Seg& s, int warp, int lane, float* scratch_m,
                           float* scratch_w) {
    const int k0 = share_of(p, s.unit_begin), k1 = share_of(p, s.unit_begin + s.n_unit - 1);
    const int nseg = k1 - k0 + 1;
    const bool k0_first = share_begin(p, k0) == s.unit_begin;
    auto slot = [&](int c) -> size_t { return (size_t)(c == 0 ? part_slot(k0, k0_first) : part_slot(k0 + c, true)); };
    const int row0 = (s.b * p.Hq + s.g * p.group) * p.S_q;
    constexpr int PER = D / 32;
    constexpr int R = NP / 4;  // rows per warp at most
    // ---- (1) M and W of every row of this warp
    float M[R], W[R];
#pragma unroll
    for (int i = 0; i < R; ++i) { M[i] = -INFINITY; W[i] = 0.f; }
    for (int c0 = 0; c0 < nseg; c0 += 32) {
        const int c = c0 + lane;
        float lv[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = warp + 4 * i;
            lv[i] = (c < nseg && r < p.rows) ? __ldcg(p.part_lse + slot(c) * NP + r) : -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float mx = lv[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_new = fmaxf(M[i], mx);
            float e = (lv[i] == -INFINITY) ? 0.f : __expf(lv[i] - m_new);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
            W[i] = (M[i] == -INFINITY ? 0.f : W[i] * __expf(M[i] - m_new)) + e;
            M[i] = m_new;
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int r = warp + 4 * i;
        if (lane == 0 && r < p.rows) {
            scratch_m[r] = M[i];
            scratch_w[r] = 1.f / W[i];
            if (p.lse) p.lse[row0 + r] = M[i] + __logf(W[i]);
        }
    }
    __syncwarp();
    // ---- (2) O = sum_c e^{LSE_c - M} O_c / W
    float acc[R][PER];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[i][e] = 0.f;
    // loads of CB partials for all rows are issued before any of them is used (the cache-global
    // loads are ordered, so program order decides how many are in flight)
    constexpr int CB = NP <= 32 ? 2 : 1;
    for (int c0 = 0; c0 < nseg; c0 += CB) {
        float lv[CB][R];
        float ov[CB][R][PER];
#pragma unroll
        for (int u = 0; u < CB; ++u) {
            const int c = c0 + u;
            const size_t sl = slot(c < nseg ? c : 0);
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = warp + 4 * i;
                lv[u][i] = -INFINITY;
#pragma unroll
                for (int e = 0; e < PER; ++e) ov[u][i][e] = 0.f;
                if (c < nseg && r < p.rows) {
                    lv[u][i] = __ldcg(p.part_lse + sl * NP + r);
                    const float* src = p.part_o + (sl * NP + r) * D + lane * PER;
                    if (PER == 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
                        ov[u][i][0] = v.x; ov[u][i][1 % PER] = v.y; ov[u][i][2 % PER] = v.z; ov[u][i][3 % PER] = v.w;
                    } else {
                        const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
                        ov[u][i][0] = v.x; ov[u][i][1 % PER] = v.y;
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < CB; ++u)
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = warp + 4 * i;
                if (r < p.rows) {
                    const float w = lv[u][i] == -INFINITY ? 0.f : __expf(lv[u][i] - scratch_m[r]) * scratch_w[r];
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[i][e] += w * ov[u][i][e];
                }
            }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int r = warp + 4 * i;
        if (r < p.rows) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + (size_t)(row0 + r) * D + lane * PER;
            if (PER == 4)
                *reinterpret_cast<uint2*>(dst) =
                    make_uint2(pack_bf16x2(acc[i][0], acc[i][1 % PER]), pack_bf16x2(acc[i][2 % PER], acc[i][3 % PER]));
            else
                *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[i][0], acc[i][1 % PER]);
        }
    }
}

template <int D, int NP, bool ALIBI>
__global__ void __launch_bounds__(NTHREADS, DCfg<D, NP>::CTAS) attn_decode_kernel(const __grid_constant__ DecodeParams p) {
    using C = DCfg<D, NP>;
    static_assert(sizeof(DShared<NP>) <= C::CTL, "control block");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned
    DShared<NP>* sh = reinterpret_cast<DShared<NP>*>(smem + C::OFF_CTL);
    const uint32_t s_kv = smem_u32(smem + C::OFF_KV);
    // ring position of K (item 2n) and V (item 2n + 1) of the CTA's tile n
    auto slot_of = [](int item) { return item % C::SLOTS; };
    auto parity_of = [](int item) { return (uint32_t)((item / C::SLOTS) & 1); };
    const uint32_t s_z = smem_u32(smem + C::OFF_Z);
    const uint32_t s_q = smem_u32(smem + C::OFF_Q);
    const uint32_t s_p = smem_u32(smem + C::OFF_P);
    auto bar = [&](int b) { return smem_u32(&sh->bar[b]); };
    const Watch wd{&sh->abort, p.err, p.watchdog_ns};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int k = blockIdx.x;
    const long long share0 = share_begin(p, k), share1 = share_begin(p, k + 1);
    const int n_tiles = (int)(share1 - share0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i == B_PFULL || i == B_PFULL + 1) ? 128u : 1u);
        sh->abort = 0;
        sh->flag = 0;
        fence_barrier_init();
    }
    if (C::ZERO) {  // zero block standing in for V^T rows 64..127 when d = 64
        for (int i = threadIdx.x; i < C::ZERO / 16; i += NTHREADS)
            reinterpret_cast<uint4*>(smem + C::OFF_Z)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sh->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == WARP_PRODUCER && lane == 0) {
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    // the merge kernel, launched as a programmatic dependent of this grid, may be scheduled
    // from here on: it waits for this grid's completion before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int n = 0, j = 0, items = 0, q_loaded = 0;
            bool ok = true;
            // the next K or V tile into the next slot, once its previous occupant has been read
            auto load_kv = [&](const CUtensorMap* tm, int key, int bkv) -> bool {
                const int sl = slot_of(items);
                if (items >= C::SLOTS && !wait_bounded(bar(B_EMPTY + sl), parity_of(items) ^ 1u, wd, ERR_PRODUCER))
                    return false;
                mbar_arrive_expect_tx(bar(B_FULL + sl), C::TB);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(s_kv + sl * C::TB + c * C::SUB, tm, bar(B_FULL + sl), c * 64, key, bkv);
                ++items;
                return true;
            };
            for (long long i = share0; i < share1 && ok; ++j) {
                const Seg s = seg_at(p, i, share1);
                i += s.count;
                if (j >= 2 && !(ok = wait_bounded(bar(B_QEMPTY + (j & 1)), ((j >> 1) - 1) & 1, wd, ERR_PRODUCER)))
                    break;
                mbar_arrive_expect_tx(bar(B_QFULL + (j & 1)), C::QT);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(s_q + (j & 1) * C::QT + c * C::QB, &p.tm_q, bar(B_QFULL + (j & 1)), c * 64,
                                (s.b * p.Hq + s.g * p.group) * p.S_q);
                q_loaded = j + 1;
                const int bkv = s.b * p.Hkv + s.g;
                for (int q = 0; q < s.count && ok; ++q, ++n) {
                    const int key = (s.tile0 + (ALIBI ? s.count - 1 - q : q)) * BN;
                    ok = load_kv(&p.tm_k, key, bkv) && load_kv(&p.tm_v, key, bkv);
                }
            }
            if (sh->abort) {  // let the copies in flight land before the CTA exits
                for (int jj = max(0, q_loaded - 2); jj < q_loaded; ++jj)
                    drain_wait(bar(B_QFULL + (jj & 1)), (jj >> 1) & 1, wd);
                for (int it = max(0, items - C::SLOTS); it < items; ++it)
                    drain_wait(bar(B_FULL + slot_of(it)), parity_of(it), wd);
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer (lane 0) + V tail zeroing (warp)
        constexpr uint32_t idesc_qk = idesc_bf16_f32_ab(BN, NP, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32_ab(BN, NP, true, false);
        // V^T as an MN-major A operand: d is contiguous; the second 64-row block of d
        // (or the zero block when d = 64) sits LBO bytes after the first
        auto v_lbo = [&](int st) -> uint32_t {
            return D == 128 ? (uint32_t)C::SUB : (uint32_t)(s_z - (s_kv + st * C::TB));
        };
        int last_bar = -1, last_par = 0;  // the last commit (drained after an abort)
        // QK of the CTA's tile n at walk position w (lane 0 only)
        auto issue_qk = [&](int n, const Walk& w) -> bool {
            const int st = slot_of(2 * n);
            if (w.q == 0 && !wait_bounded(bar(B_QFULL + (w.j & 1)), (w.j >> 1) & 1, wd, ERR_MMA)) return false;
            if (!wait_bounded(bar(B_FULL + st), parity_of(2 * n), wd, ERR_MMA)) return false;
            tc_fence_after();
            const uint32_t t_s = tmem + C::TMEM_S + (n & 1) * NP;
            const uint32_t sq = s_q + (w.j & 1) * C::QT;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t a = s_kv + st * C::TB + (kk >> 2) * C::SUB + (kk & 3) * 32;
                const uint32_t bq = sq + (kk >> 2) * C::QB + (kk & 3) * 32;
                mma_ss(t_s, sdesc_sw128(a, 16, 1024), sdesc_sw128(bq, 16, 1024), idesc_qk, kk > 0);
            }
            mma_commit(bar(B_SFULL + (n & 1)));
            mma_commit(bar(B_EMPTY + st));
            last_bar = B_SFULL + (n & 1);
            last_par = (n >> 1) & 1;
            if (w.q == w.s.count - 1) mma_commit(bar(B_QEMPTY + (w.j & 1)));
            return true;
        };
        Walk wq = walk_begin(p, share0, share1);  // tile of the next QK
        Walk wp = wq;                             // tile of the next PV
        bool ok = true;
        if (lane == 0 && wq.valid) ok = issue_qk(0, wq);
        walk_next(p, wq, share1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // The whole warp runs the loop (the exit is warp-uniform); lane 0 waits and issues.
        for (int n = 0; n < n_tiles && ok; ++n) {
            const int st = slot_of(2 * n + 1);  // V of tile n
            if (lane == 0) {
                if (wq.valid) ok = issue_qk(n + 1, wq);  // S^T buffer (n+1)&1 was released before PV(n-1)
                if (ok) ok = wait_bounded(bar(B_PFULL + (n & 1)), (n >> 1) & 1, wd, ERR_MMA);
                if (ok) ok = wait_bounded(bar(B_FULL + st), parity_of(2 * n + 1), wd, ERR_MMA);
            }
            walk_next(p, wq, share1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const int tile = wp.s.tile0 + (ALIBI ? wp.s.count - 1 - wp.q : wp.q);
            const int tail = wp.s.L % BN;
            if (tail != 0 && tile == (wp.s.L - 1) / BN) {
                // a sequence's last cache tile: zero the V rows at and past its length.  Every
                // lane observes the completed copy itself (the phase cannot advance before this PV).
                const bool seen = lane == 0 || wait_bounded(bar(B_FULL + st), parity_of(2 * n + 1), wd, ERR_MMA);
                if (!__all_sync(0xffffffffu, seen)) {
                    ok = false;
                    break;
                }
                uint8_t* vt = smem + C::OFF_KV + st * C::TB;
                const int nbytes = (BN - tail) * 128;
                for (int c = 0; c < D / 64; ++c)
                    for (int x = lane * 16; x < nbytes; x += 32 * 16)
                        *reinterpret_cast<uint4*>(vt + c * C::SUB + tail * 128 + x) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t t_o = tmem + C::TMEM_O;
                const uint32_t pb = s_p + (n & 1) * 2 * C::PB;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t a = s_kv + st * C::TB + kk * 16 * 128;  // 16 keys of 128-byte rows
                    const uint32_t bp = pb + (kk >> 2) * C::PB + (kk & 3) * 32;
                    mma_ss(t_o, sdesc_sw128(a, v_lbo(st), 1024), sdesc_sw128(bp, 16, 1024), idesc_pv,
                           (wp.q > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_EMPTY + st));
                mma_commit(bar(B_PFREE + (n & 1)));
                last_bar = B_PFREE + (n & 1);
                last_par = (n >> 1) & 1;
            }
            walk_next(p, wp, share1);
        }
        if (lane == 0 && sh->abort && last_bar >= 0) drain_wait(bar(last_bar), last_par, wd);
    } else {
        // ------------------------------------------------------------ softmax + epilogue (warps 0-3)
        // Every thread runs the same sequence of named barriers whatever happens: waits are
        // per thread and bounded, and after an abort they return at once and the remaining
        // tiles are computed on whatever is in memory (the error word is set; outputs are
        // then undefined), so no barrier is ever left incomplete.
        const int t = threadIdx.x;  // key within the tile == tensor-memory lane; d index of O^T
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        auto wait = [&](int b_, uint32_t parity) { wait_bounded(bar(b_), parity, wd, ERR_SOFTMAX); };
        // PV(m) done.  A parity wait only tells the last two phases apart, so it must never run
        // more than one phase ahead of the barrier: PFREE[m & 1] completes once per PV of that
        // parity, and this thread has already waited for PV(m - 2) on it (tile m's wait for its
        // P^T buffer), whereas a barrier completing on every PV could still be two PVs behind.
        auto wait_pv = [&](int m) { wait(B_PFREE + (m & 1), (m >> 1) & 1); };
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o);
        const bool sliding = p.kind == ATTN_MASK_CAUSAL_SLIDING;
        float lp[NP];  // this thread's share of every row's sum
        int n = 0;     // the CTA's tile counter
        int j = 0;     // stretch counter
        for (long long i = share0; i < share1; ++j) {
            const Seg s = seg_at(p, i, share1);
            i += s.count;
            const int row0 = (s.b * p.Hq + s.g * p.group) * p.S_q;
            // tightest bounds over the valid rows: a tile inside [max_lo, min_hi] needs no mask
            const int max_lo = sliding ? s.L - 1 - p.window : 0;
            const int min_hi = p.kind == ATTN_MASK_FULL ? s.L - 1 : s.L - p.S_q;
            if (t < NP) {
                int lo = 0, hi = s.L - 1;
                if (t < p.rows && p.kind != ATTN_MASK_FULL) {
                    const int pos = s.L - p.S_q + t % p.S_q;  // position of this query row
                    hi = pos;
                    if (sliding) lo = max(0, pos - p.window);
                }
                sh->lo[t] = lo;
                sh->hi[t] = hi;
                sh->m[t] = -INFINITY;
                if constexpr (ALIBI) {  // bias -m_a |t_row - j| in log2 units
                    const int rr = t < p.rows ? t : 0;
                    sh->bm[t] = p.alibi[s.g * p.group + rr / p.S_q] * 1.4426950408889634f;
                    sh->bp[t] = (float)(s.L - p.S_q + rr % p.S_q);
                }
            }
#pragma unroll
            for (int r = 0; r < NP; ++r) lp[r] = 0.f;
            named_bar_sync(1, 128);
            for (int q = 0; q < s.count; ++q, ++n) {
                const int par = n & 1;
                wait(B_SFULL + par, (n >> 1) & 1);
                if (n >= 2) wait(B_PFREE + par, ((n >> 1) - 1) & 1);  // PV(n-2) is done with this P^T buffer
                tc_fence_after();
                // with ALiBi the stretch runs from its newest key tile down (the bias falls with
                // the distance from the row's position, so the running max is set early)
                const int tile = s.tile0 + (ALIBI ? s.count - 1 - q : q);
                const int jkey = tile * BN + t;  // this thread's key
                const bool full = tile * BN >= max_lo && tile * BN + BN - 1 <= min_hi;
                const uint32_t t_s = t_lane + C::TMEM_S + par * NP;
                const int kk = t & 63;
                // this thread's column of the P^T buffer: K-major, 128B swizzle (16-byte chunk kk / 8
                // of row r sits at chunk (kk / 8) ^ (r mod 8)), the two bytes of key kk
                uint8_t* const pcol = smem + C::OFF_P + par * 2 * C::PB + (t >> 6) * C::PB + (kk & 7) * 2;
                const int kc = kk >> 3;
                float ts[NP];  // this tile's share of every row's sum
                // P = exp2(s * scale * log2 e - m) against the running max m -> bf16 P^T; returns
                // whether an allowed score exceeds m by more than the threshold.  A chunk's columns
                // are all loaded before one wait; masked scores become -inf (ex2 gives 0).  Plain
                // shared stores: the proxy fence before the P-full arrival orders them for the MMA.
                auto exp_pass = [&](auto full_c) -> bool {
                    constexpr bool FULL = decltype(full_c)::value;
                    constexpr int CH = NP < 32 ? NP : 32;  // columns per tensor-memory wait
                    float xmax = -INFINITY;
#pragma unroll
                    for (int c0 = 0; c0 < NP; c0 += CH) {
                        uint32_t v[CH];
                        float mr[CH];
                        tmem_ld16_at<0>(t_s + c0, v);
                        if constexpr (CH == 32) tmem_ld16_at<16>(t_s + c0 + 16, v);
#pragma unroll
                        for (int e = 0; e < CH; e += 4) {
                            const float4 m4 = *reinterpret_cast<const float4*>(sh->m + c0 + e);
                            mr[e] = m4.x; mr[e + 1] = m4.y; mr[e + 2] = m4.z; mr[e + 3] = m4.w;
                        }
                        if constexpr (ALIBI) {  // fold the bias into the subtracted max
#pragma unroll
                            for (int e = 0; e < CH; ++e)
                                mr[e] = fmaf(sh->bm[c0 + e], fabsf(sh->bp[c0 + e] - (float)jkey), mr[e]);
                        }
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < CH; e += 2) {
                            const int r = c0 + e;
                            float x0 = fmaf(__uint_as_float(v[e]), sl2, -mr[e]);
                            float x1 = fmaf(__uint_as_float(v[e + 1]), sl2, -mr[e + 1]);
                            if constexpr (!FULL) {
                                x0 = (jkey >= sh->lo[r] && jkey <= sh->hi[r]) ? x0 : -INFINITY;
                                x1 = (jkey >= sh->lo[r + 1] && jkey <= sh->hi[r + 1]) ? x1 : -INFINITY;
                            }
                            xmax = fmax3(xmax, x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            ts[r] = p0;
                            ts[r + 1] = p1;
                            const uint32_t pk = pack_bf16x2(p0, p1);
                            *reinterpret_cast<uint16_t*>(pcol + r * 128 + ((kc ^ (r & 7)) << 4)) = (uint16_t)pk;
                            *reinterpret_cast<uint16_t*>(pcol + (r + 1) * 128 + ((kc ^ ((r + 1) & 7)) << 4)) =
                                (uint16_t)(pk >> 16);
                        }
                    }
                    return xmax > RESCALE_THRESHOLD;
                };
                auto exp_pass_tile = [&]() -> bool {
                    return full ? exp_pass(std::true_type{}) : exp_pass(std::false_type{});
                };
                if (named_bar_or(1, 128, exp_pass_tile())) {
                    // ---- a row's max grew (always on a unit's first tile): exact masked tile maxima,
                    // new running maxima and rescale factors, then P again.  Every reader of the
                    // previous flag has passed the barrier above.
                    if (t == 0) sh->flag = 0;
#pragma unroll
                    for (int c = 0; c < NP / 16; ++c) {
                        uint32_t v[16];
                        tmem_ld16(t_s + c * 16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int r = c * 16 + e;
                            float sv = __uint_as_float(v[e]);
                            if constexpr (ALIBI)  // log2 units with the bias
                                sv = fmaf(sv, sl2, -sh->bm[r] * fabsf(sh->bp[r] - (float)jkey));
                            if (!full && !(jkey >= sh->lo[r] && jkey <= sh->hi[r])) sv = -INFINITY;
                            const int mx = __reduce_max_sync(0xffffffffu, ordered(sv));
                            if (lane == 0) sh->wmax[warp][r] = mx;
                        }
                    }
                    named_bar_sync(1, 128);
                    if (t < NP) {
                        const int k4 = max(max(sh->wmax[0][t], sh->wmax[1][t]), max(sh->wmax[2][t], sh->wmax[3][t]));
                        const float tmax = ALIBI ? unordered(k4) : unordered(k4) * sl2;  // -inf stays -inf
                        const float m_old = sh->m[t];
                        const bool grow = tmax > m_old + RESCALE_THRESHOLD;  // true on a row's first finite max
                        const float m_new = grow ? tmax : m_old;
                        sh->m[t] = m_new;
                        sh->alpha[t] = grow ? ex2(m_old - m_new) : 1.f;
                        if (grow && m_old != -INFINITY) sh->flag = 1;
                    }
                    named_bar_sync(1, 128);
                    if (sh->flag) {
                        // scale the sums and, once PV(n-1) (same unit: m_old was finite) is done, O^T
#pragma unroll
                        for (int r = 0; r < NP; ++r) lp[r] *= sh->alpha[r];
                        wait_pv(n - 1);
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < NP / 16; ++c) {
                            uint32_t o[16];
                            tmem_ld16(t_lane + C::TMEM_O + c * 16, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * sh->alpha[c * 16 + e]);
                            tmem_st16(t_lane + C::TMEM_O + c * 16, o);
                        }
                        tmem_wait_st();
                    }
                    exp_pass_tile();  // cannot exceed now (every row's m is at least its tile max)
                }
#pragma unroll
                for (int r = 0; r < NP; ++r) lp[r] += ts[r];
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(B_PFULL + par));
            }
            // ---- end of the stretch: its last PV (tile n - 1) -> O, or a partial result
            wait_pv(n - 1);
            tc_fence_after();
#pragma unroll
            for (int r = 0; r < NP; ++r) {
                float v = lp[r];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) sh->lsum[warp][r] = v;
            }
            named_bar_sync(1, 128);
            if (t < NP) {
                const float l = (sh->lsum[0][t] + sh->lsum[1][t]) + (sh->lsum[2][t] + sh->lsum[3][t]);
                sh->inv_l[t] = l > 0.f ? 1.f / l : 0.f;
                sh->lse[t] = l > 0.f ? (sh->m[t] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
            named_bar_sync(1, 128);
            const size_t slot = (size_t)part_slot(k, j == 0);
#pragma unroll
            for (int c = 0; c < NP / 16; ++c) {
                uint32_t o[16];
                tmem_ld16(t_lane + C::TMEM_O + c * 16, o);
                tmem_wait_ld();
                if (t < D) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = c * 16 + e;
                        if (r < p.rows) {
                            const float val = __uint_as_float(o[e]) * sh->inv_l[r];
                            if (s.whole) out[(size_t)(row0 + r) * D + t] = __float2bfloat16_rn(val);
                            else p.part_o[(slot * NP + r) * D + t] = val;
                        }
                    }
                }
            }
            if (t < p.rows) {
                if (s.whole) {
                    if (p.lse) p.lse[row0 + t] = sh->lse[t];
                } else {
                    p.part_lse[slot * NP + t] = sh->lse[t];
                }
            }
            // O^T has been read: the next PV into it follows this CTA's next PFULL arrival
            tc_fence_before();
            if (!s.whole && !p.defer_merge) {
                __threadfence();
                named_bar_sync(1, 128);
                if (t == 0) {
                    const int nseg = share_of(p, s.unit_begin + s.n_unit - 1) - share_of(p, s.unit_begin) + 1;
                    sh->is_last =
                        atomicInc(p.counters + s.b * p.Hkv + s.g, (unsigned)(nseg - 1)) == (unsigned)(nseg - 1);
                }
                named_bar_sync(1, 128);
                if (sh->is_last) {
                    __threadfence();
                    merge_unit<D, NP>(p, s, warp, lane, sh->alpha, sh->lse);
                }
                named_bar_sync(1, 128);  // alpha / lse are the merge's scratch; the next stretch resets m
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Merge of the split units as a kernel of its own (the decode kernel ran with defer_merge):
// warp w of CTA x takes packed row 4 (x mod R) + w of split unit x / R, R = ceil(rows / 4).
//   M = max_c LSE_c, W = sum_c e^{LSE_c - M}, O = sum_c e^{LSE_c - M} O_c / W, LSE = M + ln W
// over the unit's partials c (each normalised by its own sum).  Lane l owns d components
// [l D/32, (l+1) D/32).  Lane c loads LSE_c (c < 32) while the O values of the first PF
// partials are already in flight, so a unit of up to PF partials costs one round trip to L2.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const __grid_constant__ DecodeMergeParams p) {
    // launched as a programmatic dependent of the decode kernel: wait for that grid to complete
    // (its partial results written and visible); a no-op when launched without the attribute
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int PER = D / 32;
    constexpr int PF = 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_unit = (p.rows + 3) >> 2;
    const int u = blockIdx.x / per_unit, r = (blockIdx.x - u * per_unit) * 4 + warp;
    if (u >= p.n_split || r >= p.rows) return;  // whole warps
    const int4 e = p.list[u];
    const int b = e.x, g = e.y, k0 = e.z, nseg = e.w >> 1;
    const bool k0_first = (e.w & 1) != 0;
    auto slot = [&](int c) -> size_t { return (size_t)(c == 0 ? 2 * k0 + (k0_first ? 0 : 1) : 2 * (k0 + c)); };
    auto lse_of = [&](int c) { return __ldcg(p.part_lse + slot(c) * p.np + r); };
    auto load_o = [&](int c, float (&o)[PER]) {
        const float* src = p.part_o + (slot(c) * p.np + r) * D + lane * PER;
        if constexpr (PER == 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
            o[0] = x.x; o[1 % PER] = x.y; o[2 % PER] = x.z; o[3 % PER] = x.w;
        } else {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
            o[0] = x.x; o[1 % PER] = x.y;
        }
    };
    const float l0 = lane < nseg ? lse_of(lane) : -INFINITY;
    float ov[PF][PER];
#pragma unroll
    for (int v = 0; v < PF; ++v) {
#pragma unroll
        for (int q = 0; q < PER; ++q) ov[v][q] = 0.f;
        if (v < nseg) load_o(v, ov[v]);
    }
    float M = l0;
    for (int c = lane + 32; c < nseg; c += 32) M = fmaxf(M, lse_of(c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float W = l0 == -INFINITY ? 0.f : __expf(l0 - M);
    for (int c = lane + 32; c < nseg; c += 32) {
        const float lv = lse_of(c);
        W += lv == -INFINITY ? 0.f : __expf(lv - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    const float inv_w = W > 0.f ? 1.f / W : 0.f;
    const float w0 = l0 == -INFINITY ? 0.f : __expf(l0 - M) * inv_w;  // weight of partial `lane`
    // the weight of partial c (uniform over the warp)
    auto weight = [&](int c) -> float {
        if (c < 32) return __shfl_sync(0xffffffffu, w0, c);
        const float lv = lse_of(c);
        return lv == -INFINITY ? 0.f : __expf(lv - M) * inv_w;
    };
    float acc[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) acc[q] = 0.f;
#pragma unroll
    for (int v = 0; v < PF; ++v) {
        const float w = weight(v);  // 0 past nseg (lane v >= nseg holds l0 = -inf)
#pragma unroll
        for (int q = 0; q < PER; ++q) acc[q] = fmaf(w, ov[v][q], acc[q]);
    }
    for (int c0 = PF; c0 < nseg; c0 += PF) {
#pragma unroll
        for (int v = 0; v < PF; ++v) {
#pragma unroll
            for (int q = 0; q < PER; ++q) ov[v][q] = 0.f;
            if (c0 + v < nseg) load_o(c0 + v, ov[v]);
        }
#pragma unroll
        for (int v = 0; v < PF; ++v) {
            const float w = c0 + v < nseg ? weight(c0 + v) : 0.f;
#pragma unroll
            for (int q = 0; q < PER; ++q) acc[q] = fmaf(w, ov[v][q], acc[q]);
        }
    }
    const size_t row = (size_t)(b * p.Hq + g * p.group) * p.S_q + r;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + row * D + lane * PER;
#pragma unroll
    for (int q = 0; q < PER; ++q) dst[q] = __float2bfloat16_rn(acc[q]);
    if (lane == 0 && p.lse) p.lse[row] = W > 0.f ? M + __logf(W) : -INFINITY;
}

template <int D, int NP, bool ALIBI>
cudaError_t launch_one(const DecodeParams& p, cudaStream_t stream) {
    using C = DCfg<D, NP>;
    cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(attn_decode_kernel<D, NP, ALIBI>), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attn_decode_kernel<D, NP, ALIBI><<<p.n_cta, NTHREADS, C::SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

template <int D, int NP>
cudaError_t launch(const DecodeParams& p, cudaStream_t stream) {
    return p.alibi ? launch_one<D, NP, true>(p, stream) : launch_one<D, NP, false>(p, stream);
}

}  // namespace

cudaError_t launch_decode_merge(const DecodeMergeParams& p, int d, cudaStream_t stream) {
    if (p.n_split <= 0) return cudaSuccess;
    // a programmatic dependent launch: the grid is set up while the decode kernel still runs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_split * ((p.rows + 3) / 4)));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (d == 128) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, p);
    if (d == 64) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<64>, p);
    return cudaErrorInvalidValue;
}

// CTAs of the persistent grid per multiprocessor for a head width and packed-row width.
int decode_ctas_per_sm(int d, int np) {
    if (d == 64) return np == 16 ? DCfg<64, 16>::CTAS : np == 32 ? DCfg<64, 32>::CTAS : DCfg<64, 64>::CTAS;
    return np == 16 ? DCfg<128, 16>::CTAS : np == 32 ? DCfg<128, 32>::CTAS : DCfg<128, 64>::CTAS;
}

cudaError_t launch_decode(const DecodeParams& p, int d, int np, cudaStream_t stream) {
    if (p.n_cta <= 0 || p.total_tiles <= 0) return cudaSuccess;
    if (d == 128) {
        if (np == 16) return launch<128, 16>(p, stream);
        if (np == 32) return launch<128, 32>(p, stream);
        if (np == 64) return launch<128, 64>(p, stream);
    } else if (d == 64) {
        if (np == 16) return launch<64, 16>(p, stream);
        if (np == 32) return launch<64, 32>(p, stream);
        if (np == 64) return launch<64, 64>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace attn
