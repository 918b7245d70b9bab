// Backward pass of the attention for sm_103a (bf16 in and out, fp32 accumulation).
//
// The gradients of the forward definition (the plain derivative: the pages describe
// the tiled forward as exact and used for training, "Transformer 演进与变体"
// (ai.icyfenix.cn), section Flash Attention, and give no backward formulas):
//
//   P_ij = exp(s_ij - LSE_i),  D_i = dO_i . O_i,  dS_ij = P_ij (dO_i . v_j - D_i)
//   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i
//
// (dK and dV summed over the query heads of each kv head).  P is recomputed from the
// saved LSE, tile by tile, as the forward computed it; nothing of size S x S is stored.
//
//   bwd_prep        : -D_i and -LSE_i log2(e) into padded per-head vectors (one warp per row).
//   attn_bwd_dq     : one CTA per forward work item (128 query rows of one head).  For
//                     each allowed key tile: S = Q K^T and dP = dO V^T (tcgen05, fp32 in
//                     tensor memory), dS = P (dP - D) in bf16 over dP, and dQ += dS K with
//                     dS read from tensor memory.
//   attn_bwd_dkdv   : one CTA per key tile of one kv head, over the query tiles of every
//                     query head of the group that see it.  S^T = K Q^T and dP^T = V dO^T,
//                     P^T and dS^T in bf16 over them, dV += P^T dO and dK += dS^T Q.
//
// Both kernels: warps 0-7 compute (warpgroup h owns columns 64h .. 64h+63 of the 128 x 128
// score tile, one thread per tensor-memory lane), warp 8 loads with TMA, warp 9 issues the
// MMAs.  The score products are full 128 x 128 x 16 instructions (a 64-column product costs
// the tensor core as long as a 128-column one); the element-wise work runs in two steps --
// P from S while dP is still being computed, then dS -- and each kernel orders its MMAs so
// that the next tile's S is computed while the warps work on the current one.  tcgen05 MMAs
// of one thread run in issue order, which protects every tensor-memory column that a later
// product overwrites.
//
// Every mbarrier wait is bounded; the compute warps run the same sequence of named
// barriers whatever happens (a wait that ran out returns at once from then on), and the
// producer and MMA threads drain their copies and products before the CTA exits.
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_once.h"
#include "kernels.h"
#include "sm103_ptx.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int BT = 128;         // rows / keys per tile
constexpr int HALF = 64;        // columns per half tile
constexpr int NCOMPUTE = 256;   // two warpgroups
constexpr int NTHREADS = NCOMPUTE + 64;
constexpr int WARP_PRODUCER = 8;
constexpr int WARP_MMA = 9;
constexpr float LOG2E = 1.4426950408889634f;
enum : int { ERR_PRODUCER = 1, ERR_MMA = 2, ERR_COMPUTE = 4 };

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

// 1-D bulk copy global -> shared, completing on an mbarrier (both addresses 16-byte aligned,
// bytes a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Allowed key interval [lo, hi] of query row i, and the query interval of key j: the whole mask for
// the interval kinds, the window part of it for local + global (whose global rows and columns the
// kernels add as bits).
__device__ __forceinline__ void row_band(int kind, int window, long S, long i, long* lo, long* hi) {
    *lo = 0;
    *hi = S - 1;
    if (kind == ATTN_MASK_CAUSAL) *hi = i;
    else if (kind == ATTN_MASK_CAUSAL_SLIDING) { *lo = i - window; *hi = i; }
    else if (kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_LOCAL_GLOBAL) { *lo = i - window; *hi = i + window; }
    if (*hi > S - 1) *hi = S - 1;
}
__device__ __forceinline__ void key_band(int kind, int window, long S, long j, long* lo, long* hi) {
    *lo = 0;
    *hi = S - 1;
    if (kind == ATTN_MASK_CAUSAL) *lo = j;
    else if (kind == ATTN_MASK_CAUSAL_SLIDING) { *lo = j; *hi = j + window; }
    else if (kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_LOCAL_GLOBAL) { *lo = j - window; *hi = j + window; }
    if (*hi > S - 1) *hi = S - 1;
}

// In-tile allowed columns [a0, a1] (clamped to [-1, BT]) of an interval [lo, hi] and tile start c0.
__device__ __forceinline__ void tile_interval(long lo, long hi, long c0, int* a0, int* a1) {
    *a0 = (int)max(-1L, min((long)BT, lo - c0));
    *a1 = (int)max(-1L, min((long)BT, hi - c0));
}

// Bits of the in-tile columns [32k, 32k + 32) that lie inside [a0, a1].
__device__ __forceinline__ uint32_t interval_word(int a0, int a1, int k) {
    const int lo = max(a0 - 32 * k, 0), hi = min(a1 - 32 * k + 1, 32);  // [lo, hi)
    if (hi <= lo) return 0u;
    const uint32_t up = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
    return up & ~((1u << lo) - 1u);
}

// Whether position x is a global token (local + global): bit x % 32 of word x / 32 of the
// per-tile global bits (4 words per 128 positions).
__device__ __forceinline__ bool is_global_pos(const unsigned* gbits, long x) {
    return (__ldg(gbits + (x >> 5)) >> (x & 31)) & 1u;
}

// Local + global, a tile that is not FULL: the allowed columns of the warpgroup's half h as two
// words of bits (columns 64h .. 64h + 31, then 64h + 32 .. 64h + 63) -- the window interval
// [a0, a1] of the thread's own row (or column) plus the global positions among the tile's
// columns (or rows), gb = the tile's four words.  An own position that is global has the
// interval [0, S - 1] already.
__device__ __forceinline__ uint2 lg_half_bits(int a0, int a1, const unsigned* gb, int h) {
    return make_uint2(interval_word(a0, a1, 2 * h) | __ldg(gb + 2 * h),
                      interval_word(a0, a1, 2 * h + 1) | __ldg(gb + 2 * h + 1));
}

// ------------------------------------------------------------------ pre-pass
// -D_i = -dO_i . O_i and -LSE_i log2 e for every row, padded to whole tiles (padding rows:
// -inf and 0, so their P is 0).  A row is d/8 lanes reading 16 bytes each of O and dO; a warp
// handles PREP_ROUNDS groups of 32/(d/8) rows, with every load issued before the reductions.
constexpr int PREP_ROUNDS = 4;
constexpr int PREP_WARPS = 8;

__global__ void __launch_bounds__(PREP_WARPS * 32) bwd_prep_kernel(BwdPrepParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = p.d >> 3, rows_per_round = 32 / L;  // d = 64 or 128: 8 or 16 lanes per row
    const int sub = lane / L, lc = lane - sub * L;
    const long total = (long)p.BHq * p.S_pad;
    const long row0 = ((long)blockIdx.x * PREP_WARPS + warp) * (PREP_ROUNDS * rows_per_round);
    float acc[PREP_ROUNDS];
    uint4 o4[PREP_ROUNDS], g4[PREP_ROUNDS];
#pragma unroll
    for (int r = 0; r < PREP_ROUNDS; ++r) {
        const long row = row0 + r * rows_per_round + sub;
        o4[r] = g4[r] = make_uint4(0, 0, 0, 0);
        if (row < total) {
            const long bh = row / p.S_pad, i = row - bh * p.S_pad;
            if (i < p.S) {
                const long src = (bh * p.S + i) * p.d + lc * 8;
                o4[r] = *reinterpret_cast<const uint4*>(p.o + src);
                g4[r] = *reinterpret_cast<const uint4*>(p.dout + src);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < PREP_ROUNDS; ++r) {
        const uint32_t ow[4] = {o4[r].x, o4[r].y, o4[r].z, o4[r].w}, gw[4] = {g4[r].x, g4[r].y, g4[r].z, g4[r].w};
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            a = fmaf(__uint_as_float(ow[e] << 16), __uint_as_float(gw[e] << 16), a);
            a = fmaf(__uint_as_float(ow[e] & 0xffff0000u), __uint_as_float(gw[e] & 0xffff0000u), a);
        }
        acc[r] = a;
    }
#pragma unroll
    for (int r = 0; r < PREP_ROUNDS; ++r)
        for (int off = L >> 1; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    if (lc == 0) {
#pragma unroll
        for (int r = 0; r < PREP_ROUNDS; ++r) {
            const long row = row0 + r * rows_per_round + sub;
            if (row >= total) continue;
            const long bh = row / p.S_pad, i = row - bh * p.S_pad;
            if (i < p.S) {
                p.nd[row] = -acc[r];
                p.nlse2[row] = -p.lse[bh * p.S + i] * LOG2E;
            } else {
                p.nd[row] = 0.f;
                p.nlse2[row] = -INFINITY;
            }
        }
    }
}

// 32-column groups g0 .. g0+NG-1 of a 128-row tile in tensor memory (columns col0 + 32 g),
// times f, as bf16 into 128B-swizzled staging (64-column blocks of 128 rows x 128 B) for a
// TMA store; thread r writes row r.
template <int NG>
__device__ __forceinline__ void stage_groups(uint8_t* stage, uint32_t t_lane, uint32_t col0, int g0, int r, float f) {
#pragma unroll
    for (int k = 0; k < NG; ++k) {
        const int g = g0 + k;
        uint32_t o[32];
        tmem_ld32(t_lane + col0 + g * 32, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * f, __uint_as_float(o[2 * e + 1]) * f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int chunk = (g & 1) * 4 + q;
            uint4* dst = reinterpret_cast<uint4*>(stage + (g >> 1) * (BT * 128) + r * 128 + ((chunk ^ (r & 7)) << 4));
            *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
    }
}

// Mask forms of a tile: none (FULL), the interval [a0, a1] of in-tile columns, or column bits
// (local + global: bit c % 32 of the word of the column's 32-column chunk).
enum { MK_NONE = 0, MK_INTERVAL = 1, MK_BITS = 2 };

// Score of in-tile column c, -inf where the tile's mask form excludes it (w: the bits of the
// column's chunk).
template <int MK>
__device__ __forceinline__ float masked(uint32_t raw, int c, int a0, int a1, uint32_t w) {
    if (MK == MK_NONE) return __uint_as_float(raw);
    if (MK == MK_INTERVAL) return (c >= a0 && c <= a1) ? __uint_as_float(raw) : -INFINITY;
    return ((w >> (c & 31)) & 1u) ? __uint_as_float(raw) : -INFINITY;
}

// The element-wise work of one warpgroup on its half of a tile (columns 64h .. 64h+63 of the
// 128-column score tile; one thread per tensor-memory lane), in two steps so that the first
// can run while the tensor core still computes dP:
//   exp_pass: P = 2^(s sl2 - LSE log2 e) in fp32 registers (0 where masked), and optionally P
//             rounded to bf16 and packed two per column over the first 32 columns of the half;
//   ds_pass : dS = P (dP - D), rounded to bf16 and packed over the first 32 dP columns of the half.
// The row's (dQ kernel) or the columns' (dK/dV kernel, from shared memory) -LSE log2 e and -D
// come in through NL / ND.
struct RowConst {  // one value for every column: the thread's own query row
    float v;
    __device__ __forceinline__ float4 quad(int) const { return make_float4(v, v, v, v); }
};
struct ColVec {  // one value per column, from a 16-byte aligned shared-memory vector of 128 floats;
                 // every lane reads the same 16 bytes (one broadcast wavefront per 4 columns)
    uint32_t v;  // shared-memory address
    __device__ __forceinline__ float4 quad(int c) const {
        float4 r;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                     : "r"(v + 4u * (uint32_t)c));
        return r;
    }
};

// With AL, the ALiBi bias -m_a |i - j| joins the exponent, in log2 units: -mL |base - c| for in-tile
// column c (mL = m_a log2 e; base = the thread's own position minus the first position of the
// tile's columns, for query rows and key columns alike).
// With a bias matrix, bias.chunk(ch, b) fills b with the bf16 bits of b_ij for the 32 columns
// cb .. cb + 31 (two per word, the lower column in the low half; zero where nothing is read), issued
// before the scores are loaded; b_ij log2 e joins the exponent.
struct NoBias {
    static constexpr bool on = false;
    __device__ __forceinline__ void chunk(int, uint32_t (&)[16]) const {}
};
template <int MK, bool STORE_P, bool AL, class NL, class BV = NoBias>
__device__ __forceinline__ void exp_pass(uint32_t t_s, int h, float sl2, NL nl, int a0, int a1, uint2 mw, float mL,
                                         float base, float (&pv)[64], BV bias = BV{}) {
    const float2 sl = make_float2(sl2, sl2);
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        const int cb = h * HALF + ch * 32;
        uint32_t s[32], pk[16], bw[16];
        if constexpr (BV::on) bias.chunk(ch, bw);
        tmem_ld32(t_s + cb, s);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const int c = cb + 2 * e;
            const float4 n4 = nl.quad(c);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int k = 2 * (e + u);
                float2 add = u ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y);
                if (AL) {
                    add.x = fmaf(-mL, fabsf(base - (float)(cb + k)), add.x);
                    add.y = fmaf(-mL, fabsf(base - (float)(cb + k + 1)), add.y);
                }
                if constexpr (BV::on) {
                    const uint32_t wv = bw[k >> 1];
                    add = __ffma2_rn(make_float2(__uint_as_float(wv << 16), __uint_as_float(wv & 0xffff0000u)),
                                     make_float2(LOG2E, LOG2E), add);
                }
                const uint32_t w = ch ? mw.y : mw.x;
                const float2 x = __ffma2_rn(make_float2(masked<MK>(s[k], cb + k, a0, a1, w),
                                                        masked<MK>(s[k + 1], cb + k + 1, a0, a1, w)),
                                            sl, add);
                pv[ch * 32 + k] = ex2(x.x);
                pv[ch * 32 + k + 1] = ex2(x.y);
                if (STORE_P) pk[e + u] = pack_bf16x2(pv[ch * 32 + k], pv[ch * 32 + k + 1]);
            }
        }
        if (STORE_P) tmem_st16(t_s + h * HALF + ch * 16, pk);
    }
}

// The dQ kernel's bias reader: the thread's query row, 16-byte loads along the row (b points at the
// row's bias at the first column of the warpgroup's half; n = columns of the half inside the
// sequence, counted from there).
struct RowBias {
    static constexpr bool on = true;
    const uint16_t* b;
    int n;
    __device__ __forceinline__ void chunk(int ch, uint32_t (&w)[16]) const {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c = ch * 32 + q * 8;
            // a load that starts inside the sequence stays inside the row (the stride is a multiple of 8);
            // the row's padding past the sequence may hold anything, so those columns are zeroed here
            // (their scores are masked to -inf, and -inf + NaN would not be)
            const uint4 v = (b != nullptr && c < n) ? __ldg(reinterpret_cast<const uint4*>(b + c))
                                                    : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = c + 2 * e;
                w[4 * q + e] = (col + 1 < n) ? vw[e] : (col < n) ? (vw[e] & 0xffffu) : 0u;
            }
        }
    }
};
// The dK/dV kernel's bias reader: the thread's key column, one 2-byte load per query row (b points at
// b[first query row of the warpgroup's half][key]; ld = the row stride; n = rows inside the sequence).
struct ColBias {
    static constexpr bool on = true;
    const uint16_t* b;
    long ld;
    int n;
    __device__ __forceinline__ void chunk(int ch, uint32_t (&w)[16]) const {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int c = ch * 32 + 2 * e;
            const uint32_t lo = (b != nullptr && c < n) ? (uint32_t)__ldg(b + (long)c * ld) : 0u;
            const uint32_t hi = (b != nullptr && c + 1 < n) ? (uint32_t)__ldg(b + (long)(c + 1) * ld) : 0u;
            w[e] = lo | (hi << 16);
        }
    }
};

template <class ND>
__device__ __forceinline__ void ds_pass(uint32_t t_dp, int h, ND nd, const float (&pv)[64]) {
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        const int cb = h * HALF + ch * 32;
        uint32_t g[32], pk[16];
        tmem_ld32(t_dp + cb, g);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const float4 n4 = nd.quad(cb + 2 * e);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int k = 2 * (e + u);
                const float2 dd = __fadd2_rn(make_float2(__uint_as_float(g[k]), __uint_as_float(g[k + 1])),
                                             u ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y));
                const float2 ds = __fmul2_rn(make_float2(pv[ch * 32 + k], pv[ch * 32 + k + 1]), dd);
                pk[e + u] = pack_bf16x2(ds.x, ds.y);
            }
        }
        tmem_st16(t_dp + h * HALF + ch * 16, pk);
    }
}

// ------------------------------------------------------------------ dQ kernel
// Tensor memory: three 128-column score regions R0..R2 and dQ.  Tile n keeps S in region
// (2n) mod 3 and dP in region (2n+1) mod 3, so S of tile n+2 lands in the region that held
// dP of tile n (free once dQ(n) has read dS) and dP of tile n+1 in the region of S(n) (free
// once the compute warps have read S(n)).  S(n+2) is therefore computed while the warps work
// on tile n+1.  K has three shared-memory stages (S runs two tiles ahead), V two.
template <int D>
struct DqCfg {
    static constexpr int TB = BT * D * 2;  // one Q / dO / K / V tile
    static constexpr int SUB = BT * 128;   // one 64-column swizzled block
    static constexpr int KST = 3, VST = 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + TB;
    static constexpr int OFF_K = OFF_DO + TB;
    static constexpr int OFF_V = OFF_K + KST * TB;
    static constexpr int OFF_CTL = OFF_V + VST * TB;
    static constexpr int SMEM_ALLOC = OFF_CTL + 1024 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TMEM_DQ = 384;
};

// Barriers and why no wait can fall two phases behind (a parity wait would then hang):
//   Q_KFULL[n%3] / Q_KEMPTY[n%3], Q_VFULL[n&1] / Q_VEMPTY[n&1]: rings; a stage is refilled only after
//       its empty barrier completed for the tile two (V) or three (K) back.
//   Q_SFULL[n&1]: S(n+2) is issued only after the dQ update of tile n, i.e. after both warpgroups
//       arrived on Q_HDONE for n; alternating two barriers keeps S(n+1) and S(n+2) on different ones.
//   Q_DPFULL: dP(n+1) is issued only after Q_HDONE(n), so the warps wait at most one phase back.
//   Q_HDONE[h] (128 arrivals): the warpgroup arrives for n+1 only after Q_DPFULL(n+1), which the MMA
//       thread commits after it has seen Q_HDONE(n).
enum DqBar { Q_LOAD = 0, Q_KFULL, Q_KEMPTY = Q_KFULL + 3, Q_VFULL = Q_KEMPTY + 3, Q_VEMPTY = Q_VFULL + 2,
             Q_SFULL = Q_VEMPTY + 2, Q_DPFULL = Q_SFULL + 2, Q_HDONE, Q_DONE = Q_HDONE + 2, Q_DRAIN, Q_NBAR };
static_assert(Q_NBAR <= 24, "barrier slots");

struct BwdShared {
    uint64_t bar[24];
    uint32_t tmem_base;
    volatile int abort;
};

__device__ __forceinline__ uint32_t region_s(int n) { return (uint32_t)((2 * n) % 3) * 128u; }
__device__ __forceinline__ uint32_t region_dp(int n) { return (uint32_t)((2 * n + 1) % 3) * 128u; }

template <int D, bool AL, bool BM, bool LG>
__global__ void __launch_bounds__(NTHREADS, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    BwdShared* sh = reinterpret_cast<BwdShared*>(smem + C::OFF_CTL);
    auto bar = [&](int b) { return smem_u32(&sh->bar[b]); };
    const Watch wd{&sh->abort, p.err, p.watchdog_ns};
    const uint32_t s_q = smem_u32(smem + C::OFF_Q), s_do = smem_u32(smem + C::OFF_DO);
    const uint32_t s_k = smem_u32(smem + C::OFF_K), s_v = smem_u32(smem + C::OFF_V);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int4 w0 = p.work[2 * blockIdx.x], w1 = p.work[2 * blockIdx.x + 1];
    const int bh = w0.x, q_tile = w0.y, kv_begin = w0.z, kv_end = w0.w;
    const int full_begin = w1.x, full_end = w1.y;
    const int n_iter = kv_end - kv_begin;
    const int b = bh / p.Hq, a = bh - b * p.Hq;
    const int bkv = b * p.Hkv + a / p.group;
    // key tile of iteration it: a contiguous range, or (local + global) the query tile's list
    auto key_tile = [&](int it) { return LG ? (__ldg(p.list + kv_begin + it) & (kListFull - 1)) : kv_begin + it; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < Q_NBAR; ++i) mbar_init(bar(i), (i == Q_HDONE || i == Q_HDONE + 1) ? 128u : 1u);
        sh->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sh->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == WARP_PRODUCER && lane == 0) {
        prefetch_tmap(&p.tm_q); prefetch_tmap(&p.tm_do); prefetch_tmap(&p.tm_k); prefetch_tmap(&p.tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;

    if (warp == WARP_PRODUCER) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(Q_LOAD), 2 * C::TB);
            for (int s = 0; s < D / 64; ++s) {
                tma_load_3d(s_q + s * C::SUB, &p.tm_q, bar(Q_LOAD), s * 64, q_tile * BT, bh);
                tma_load_3d(s_do + s * C::SUB, &p.tm_do, bar(Q_LOAD), s * 64, q_tile * BT, bh);
            }
            int k_loaded = 0, v_loaded = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int row = key_tile(it) * BT, ks = it % 3, vs = it & 1;
                if (it >= 3 && !wait_bounded(bar(Q_KEMPTY + ks), (it / 3 - 1) & 1, wd, ERR_PRODUCER)) break;
                mbar_arrive_expect_tx(bar(Q_KFULL + ks), C::TB);
                for (int s = 0; s < D / 64; ++s)
                    tma_load_3d(s_k + ks * C::TB + s * C::SUB, &p.tm_k, bar(Q_KFULL + ks), s * 64, row, bkv);
                k_loaded = it + 1;
                if (it >= 2 && !wait_bounded(bar(Q_VEMPTY + vs), ((it >> 1) - 1) & 1, wd, ERR_PRODUCER)) break;
                mbar_arrive_expect_tx(bar(Q_VFULL + vs), C::TB);
                for (int s = 0; s < D / 64; ++s)
                    tma_load_3d(s_v + vs * C::TB + s * C::SUB, &p.tm_v, bar(Q_VFULL + vs), s * 64, row, bkv);
                v_loaded = it + 1;
            }
            if (sh->abort) {
                drain_wait(bar(Q_LOAD), 0, wd);
                for (int n = max(0, k_loaded - 3); n < k_loaded; ++n) drain_wait(bar(Q_KFULL + n % 3), (n / 3) & 1, wd);
                for (int n = max(0, v_loaded - 2); n < v_loaded; ++n) drain_wait(bar(Q_VFULL + (n & 1)), (n >> 1) & 1, wd);
            }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BT, BT, false);  // [128 x 128] = A[128 x d] . B[128 x d]^T
            constexpr uint32_t idesc_q = idesc_bf16_f32(BT, D, true);    // dQ += dS (tensor memory) . K (MN-major)
            const uint32_t t_dq = tmem + C::TMEM_DQ;
            auto issue_s = [&](int n) {  // S(n) = Q K(n)^T
                const uint32_t sk = s_k + (n % 3) * C::TB, d = tmem + region_s(n);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::SUB + (k & 3) * 32;
                    mma_ss(d, sdesc_sw128(s_q + off, 16, 1024), sdesc_sw128(sk + off, 16, 1024), idesc_s, k > 0);
                }
                mma_commit(bar(Q_SFULL + (n & 1)));
            };
            auto issue_dp = [&](int n) {  // dP(n) = dO V(n)^T
                const uint32_t sv = s_v + (n & 1) * C::TB, d = tmem + region_dp(n);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::SUB + (k & 3) * 32;
                    mma_ss(d, sdesc_sw128(s_do + off, 16, 1024), sdesc_sw128(sv + off, 16, 1024), idesc_s, k > 0);
                }
                mma_commit(bar(Q_DPFULL));
                mma_commit(bar(Q_VEMPTY + (n & 1)));
            };
            auto issue_dq = [&](int n, int h) {  // dQ += dS_h(n) K_h(n) (64 keys: four K=16 steps)
                const uint32_t sk = s_k + (n % 3) * C::TB, a_t = tmem + region_dp(n) + h * HALF;
#pragma unroll
                for (int k = 0; k < HALF / 16; ++k)
                    mma_ts(t_dq, a_t + k * 8, sdesc_sw128(sk + (h * HALF + k * 16) * 128, C::SUB, 1024), idesc_q,
                           (n == 0 && h == 0 && k == 0) ? 0u : 1u);
            };
            bool ok = wait_bounded(bar(Q_LOAD), 0, wd, ERR_MMA) && wait_bounded(bar(Q_KFULL), 0, wd, ERR_MMA);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                ok = wait_bounded(bar(Q_VFULL), 0, wd, ERR_MMA);
            }
            if (ok) {
                tc_fence_after();
                issue_dp(0);
                if (n_iter > 1 && (ok = wait_bounded(bar(Q_KFULL + 1), 0, wd, ERR_MMA))) {
                    tc_fence_after();
                    issue_s(1);
                }
            }
            for (int it = 0; it < n_iter && ok; ++it) {
                if (!(ok = wait_bounded(bar(Q_HDONE), it & 1, wd, ERR_MMA))) break;
                tc_fence_after();
                issue_dq(it, 0);
                if (!(ok = wait_bounded(bar(Q_HDONE + 1), it & 1, wd, ERR_MMA))) break;
                tc_fence_after();
                issue_dq(it, 1);
                mma_commit(bar(Q_KEMPTY + it % 3));
                if (it + 1 < n_iter) {
                    const int n1 = it + 1;
                    if (!(ok = wait_bounded(bar(Q_VFULL + (n1 & 1)), (n1 >> 1) & 1, wd, ERR_MMA))) break;
                    tc_fence_after();
                    issue_dp(n1);
                }
                if (it + 2 < n_iter) {
                    const int n2 = it + 2;
                    if (!(ok = wait_bounded(bar(Q_KFULL + n2 % 3), (n2 / 3) & 1, wd, ERR_MMA))) break;
                    tc_fence_after();
                    issue_s(n2);
                }
            }
            if (ok) mma_commit(bar(Q_DONE));
            if (sh->abort) {
                mma_commit(bar(Q_DRAIN));
                drain_wait(bar(Q_DRAIN), 0, wd);
            }
        }
    } else {
        // compute warps: warpgroup wg owns key columns 64 wg .. 64 wg + 63; one thread per query row
        const int wg = warp >> 2, r = (warp & 3) * 32 + lane;
        const long i = (long)q_tile * BT + r;
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const RowConst nl{p.nlse2[(size_t)bh * p.S_pad + i]}, nd{p.nd[(size_t)bh * p.S_pad + i]};
        const float sl2 = p.scale_log2;
        long lo, hi;
        row_band(p.kind, p.window, p.S, i, &lo, &hi);
        if (LG && i < p.S && is_global_pos(p.gbits, i)) { lo = 0; hi = p.S - 1; }  // a global row sees every key
        const float mL = AL ? p.alibi[a] * LOG2E : 0.f;  // ALiBi slope of this query head, log2 units
        float pv[64];
        for (int it = 0; it < n_iter; ++it) {
            const int e = LG ? __ldg(p.list + kv_begin + it) : 0;
            const int t = LG ? (e & (kListFull - 1)) : kv_begin + it;
            const bool full = LG ? (e & kListFull) != 0 : (t >= full_begin && t < full_end);
            int a0, a1;
            tile_interval(lo, hi, (long)t * BT, &a0, &a1);
            // local + global: the window interval plus the tile's global keys, as bits
            const uint2 bw = (LG && !full) ? lg_half_bits(a0, a1, p.gbits + 4 * t, wg) : make_uint2(0u, 0u);
            const float base = (float)(i - (long)t * BT);
            wait_bounded(bar(Q_SFULL + (it & 1)), (it >> 1) & 1, wd, ERR_COMPUTE);
            tc_fence_after();
            constexpr int MKP = LG ? MK_BITS : MK_INTERVAL;  // the mask form of the tiles that are not FULL
            if constexpr (BM) {  // the bias row of this query row over the warpgroup's 64 columns
                const size_t plane = (size_t)(p.bias_Bb == 1 ? 0 : b) * p.bias_Hb + (p.bias_Hb == 1 ? 0 : a);
                const long c0 = (long)t * BT + wg * HALF;
                const RowBias rb{i < p.S ? p.bias + (plane * (size_t)p.S + (size_t)i) * (size_t)p.bias_ld + c0 : nullptr,
                                 (int)min((long)HALF, (long)p.S - c0)};
                if (!full)
                    exp_pass<MKP, false, AL>(t_lane + region_s(it), wg, sl2, nl, a0, a1, bw, mL, base, pv, rb);
                else
                    exp_pass<MK_NONE, false, AL>(t_lane + region_s(it), wg, sl2, nl, a0, a1, bw, mL, base, pv, rb);
            } else {
                if (!full)
                    exp_pass<MKP, false, AL>(t_lane + region_s(it), wg, sl2, nl, a0, a1, bw, mL, base, pv);
                else
                    exp_pass<MK_NONE, false, AL>(t_lane + region_s(it), wg, sl2, nl, a0, a1, bw, mL, base, pv);
            }
            wait_bounded(bar(Q_DPFULL), it & 1, wd, ERR_COMPUTE);
            tc_fence_after();
            ds_pass(t_lane + region_dp(it), wg, nd, pv);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(Q_HDONE + wg));
        }
        // epilogue: dQ * scale -> bf16 -> swizzled staging in the Q buffer -> TMA store
        wait_bounded(bar(Q_DONE), 0, wd, ERR_COMPUTE);
        tc_fence_after();
        stage_groups<D / 64>(smem + C::OFF_Q, t_lane, C::TMEM_DQ, wg * (D / 64), r, p.scale);
        fence_proxy_async_smem();
        named_bar_sync(1, NCOMPUTE);
        if (threadIdx.x == 0 && !sh->abort) {
            for (int s = 0; s < D / 64; ++s) tma_store_3d(&p.tm_dq, s_q + s * C::SUB, s * 64, q_tile * BT, bh);
            tma_store_commit_and_wait_read();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ dK / dV kernel
// Per (head, query tile) iteration n the MMA thread issues
//     S^T(n) | dP^T(n) | dV_0(n) dV_1(n) | S^T(n+1) | dK_0(n) dK_1(n) | dP^T(n+1) | ...
// dV_h needs warpgroup h's P^T (its exp step), dK_h its dS^T (its dS step).  S^T(n+1) may
// overwrite the S^T columns once both dV halves are issued (they read P^T from there), and
// dP^T(n+1) the dP^T columns once both dK halves are; so the exp step of tile n+1 overlaps
// dK(n) and dP^T(n+1) on the tensor core.
template <int D>
struct KvCfg {
    static constexpr int TB = BT * D * 2;
    static constexpr int SUB = BT * 128;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TB;
    static constexpr int OFF_Q = OFF_V + TB;        // two stages
    static constexpr int OFF_DO = OFF_Q + 2 * TB;   // two stages
    static constexpr int OFF_VEC = OFF_DO + 2 * TB; // two stages of 128 -LSE log2 e + 128 -D
    static constexpr int OFF_CTL = OFF_VEC + 2 * 1024;
    static constexpr int SMEM_ALLOC = OFF_CTL + 1024 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TMEM_S = 0, TMEM_DP = 128, TMEM_DV = 256, TMEM_DK = 256 + D;
};

// Barriers and why no wait can fall two phases behind:
//   KV_QFULL[n&1] / KV_QEMPTY[n&1]: a Q/dO/vector stage is refilled only after the dK update of the
//       tile two back, which needs both warpgroups' KV_HDONE for it.
//   KV_SFULL: S^T(n+1) is issued only after both KV_PDONE(n); KV_DPFULL: dP^T(n+1) only after both
//       KV_HDONE(n).  A warpgroup waits for either at most one phase back.
//   KV_PDONE[h] / KV_HDONE[h] (128 arrivals each): arrivals for n+1 need KV_SFULL(n+1) / KV_DPFULL(n+1),
//       which the MMA thread commits after it has seen the arrivals for n.
enum KvBar { KV_LOAD = 0, KV_QFULL, KV_QEMPTY = KV_QFULL + 2, KV_SFULL = KV_QEMPTY + 2, KV_DPFULL, KV_PDONE,
             KV_HDONE = KV_PDONE + 2, KV_DONE = KV_HDONE + 2, KV_DRAIN, KV_NBAR };
static_assert(KV_NBAR <= 24, "barrier slots");

template <int D, bool AL, bool BM, bool LG>
__global__ void __launch_bounds__(NTHREADS, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using C = KvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    BwdShared* sh = reinterpret_cast<BwdShared*>(smem + C::OFF_CTL);
    auto bar = [&](int b) { return smem_u32(&sh->bar[b]); };
    const Watch wd{&sh->abort, p.err, p.watchdog_ns};
    const uint32_t s_k = smem_u32(smem + C::OFF_K), s_v = smem_u32(smem + C::OFF_V);
    const uint32_t s_q = smem_u32(smem + C::OFF_Q), s_do = smem_u32(smem + C::OFF_DO);
    const uint32_t s_vec = smem_u32(smem + C::OFF_VEC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int bkv = blockIdx.x / p.n_items, item = blockIdx.x - bkv * p.n_items;
    const int4 w0 = p.work[2 * item], w1 = p.work[2 * item + 1];
    const int kv_tile = w0.x, q_begin = w0.y, q_end = w0.z, full_begin = w0.w, full_end = w1.x;
    const int n_q = q_end - q_begin;
    const int n_iter = p.group * n_q;  // query heads of the group x query tiles
    const int b = bkv / p.Hkv, g = bkv - b * p.Hkv;
    auto iter_head = [&](int it) { return b * p.Hq + g * p.group + it / n_q; };
    // query tile of iteration it: a contiguous range, or (local + global) the key tile's list
    auto iter_entry = [&](int it) { return LG ? __ldg(p.list + q_begin + it % n_q) : q_begin + it % n_q; };
    auto iter_qtile = [&](int it) { return LG ? (iter_entry(it) & (kListFull - 1)) : q_begin + it % n_q; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < KV_NBAR; ++i) {
            const bool wg_bar = i == KV_PDONE || i == KV_PDONE + 1 || i == KV_HDONE || i == KV_HDONE + 1;
            mbar_init(bar(i), wg_bar ? 128u : 1u);
        }
        sh->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sh->tmem_base), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == WARP_PRODUCER && lane == 0) {
        prefetch_tmap(&p.tm_q); prefetch_tmap(&p.tm_do); prefetch_tmap(&p.tm_k); prefetch_tmap(&p.tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;

    if (warp == WARP_PRODUCER) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(KV_LOAD), 2 * C::TB);
            for (int s = 0; s < D / 64; ++s) {
                tma_load_3d(s_k + s * C::SUB, &p.tm_k, bar(KV_LOAD), s * 64, kv_tile * BT, bkv);
                tma_load_3d(s_v + s * C::SUB, &p.tm_v, bar(KV_LOAD), s * 64, kv_tile * BT, bkv);
            }
            int loaded = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int st = it & 1, bh = iter_head(it), qt = iter_qtile(it);
                if (it >= 2 && !wait_bounded(bar(KV_QEMPTY + st), ((it >> 1) - 1) & 1, wd, ERR_PRODUCER)) break;
                mbar_arrive_expect_tx(bar(KV_QFULL + st), 2 * C::TB + 1024);
                for (int s = 0; s < D / 64; ++s) {
                    tma_load_3d(s_q + st * C::TB + s * C::SUB, &p.tm_q, bar(KV_QFULL + st), s * 64, qt * BT, bh);
                    tma_load_3d(s_do + st * C::TB + s * C::SUB, &p.tm_do, bar(KV_QFULL + st), s * 64, qt * BT, bh);
                }
                const size_t v0 = (size_t)bh * p.S_pad + (size_t)qt * BT;
                bulk_load(s_vec + st * 1024, p.nlse2 + v0, 512, bar(KV_QFULL + st));
                bulk_load(s_vec + st * 1024 + 512, p.nd + v0, 512, bar(KV_QFULL + st));
                loaded = it + 1;
            }
            if (sh->abort) {
                drain_wait(bar(KV_LOAD), 0, wd);
                for (int n = max(0, loaded - 2); n < loaded; ++n) drain_wait(bar(KV_QFULL + (n & 1)), (n >> 1) & 1, wd);
            }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BT, BT, false);
            constexpr uint32_t idesc_kv = idesc_bf16_f32(BT, D, true);  // dV, dK += (tensor memory) . (MN-major)
            const uint32_t t_s = tmem + C::TMEM_S, t_dp = tmem + C::TMEM_DP;
            const uint32_t t_dv = tmem + C::TMEM_DV, t_dk = tmem + C::TMEM_DK;
            auto issue_s = [&](int n) {  // S^T(n) = K Q(n)^T
                const uint32_t sq = s_q + (n & 1) * C::TB;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::SUB + (k & 3) * 32;
                    mma_ss(t_s, sdesc_sw128(s_k + off, 16, 1024), sdesc_sw128(sq + off, 16, 1024), idesc_s, k > 0);
                }
                mma_commit(bar(KV_SFULL));
            };
            auto issue_dp = [&](int n) {  // dP^T(n) = V dO(n)^T
                const uint32_t sdo = s_do + (n & 1) * C::TB;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::SUB + (k & 3) * 32;
                    mma_ss(t_dp, sdesc_sw128(s_v + off, 16, 1024), sdesc_sw128(sdo + off, 16, 1024), idesc_s, k > 0);
                }
                mma_commit(bar(KV_DPFULL));
            };
            // acc += (tensor-memory operand of half h) . (rows 64h .. 64h+63 of the stage's tile, MN-major)
            auto issue_half = [&](uint32_t acc, uint32_t a_t, uint32_t tile, int h, bool first) {
#pragma unroll
                for (int k = 0; k < HALF / 16; ++k)
                    mma_ts(acc, a_t + h * HALF + k * 8, sdesc_sw128(tile + (h * HALF + k * 16) * 128, C::SUB, 1024),
                           idesc_kv, (first && k == 0) ? 0u : 1u);
            };
            bool ok = wait_bounded(bar(KV_LOAD), 0, wd, ERR_MMA) && wait_bounded(bar(KV_QFULL), 0, wd, ERR_MMA);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp(0);
            }
            for (int it = 0; it < n_iter && ok; ++it) {
                const int st = it & 1;
                const uint32_t sq = s_q + st * C::TB, sdo = s_do + st * C::TB;
                for (int h = 0; h < 2 && ok; ++h) {  // dV += P^T_h dO_h
                    if (!(ok = wait_bounded(bar(KV_PDONE + h), it & 1, wd, ERR_MMA))) break;
                    tc_fence_after();
                    issue_half(t_dv, t_s, sdo, h, it == 0 && h == 0);
                }
                if (!ok) break;
                if (it + 1 < n_iter) {
                    if (!(ok = wait_bounded(bar(KV_QFULL + (st ^ 1)), ((it + 1) >> 1) & 1, wd, ERR_MMA))) break;
                    tc_fence_after();
                    issue_s(it + 1);
                }
                for (int h = 0; h < 2 && ok; ++h) {  // dK += dS^T_h Q_h
                    if (!(ok = wait_bounded(bar(KV_HDONE + h), it & 1, wd, ERR_MMA))) break;
                    tc_fence_after();
                    issue_half(t_dk, t_dp, sq, h, it == 0 && h == 0);
                }
                if (!ok) break;
                mma_commit(bar(KV_QEMPTY + st));
                if (it + 1 < n_iter) issue_dp(it + 1);
            }
            if (ok) mma_commit(bar(KV_DONE));
            if (sh->abort) {
                mma_commit(bar(KV_DRAIN));
                drain_wait(bar(KV_DRAIN), 0, wd);
            }
        }
    } else {
        // compute warps: warpgroup wg owns query columns 64 wg .. 64 wg + 63; one thread per key
        const int wg = warp >> 2, t = (warp & 3) * 32 + lane;
        const long j = (long)kv_tile * BT + t;
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t t_s = t_lane + C::TMEM_S, t_dp = t_lane + C::TMEM_DP;
        const float sl2 = p.scale_log2;
        long ilo, ihi;
        key_band(p.kind, p.window, p.S, j, &ilo, &ihi);
        if (LG && j < p.S && is_global_pos(p.gbits, j)) { ilo = 0; ihi = p.S - 1; }  // a global key is seen by every row
        if (j >= p.S) { ilo = 1; ihi = 0; }  // a padding key sees no row
        float pv[64];
        for (int it = 0; it < n_iter; ++it) {
            const int st = it & 1, qt = iter_qtile(it);
            const bool full = LG ? (iter_entry(it) & kListFull) != 0 : (qt >= full_begin && qt < full_end);
            int a0, a1;
            tile_interval(ilo, ihi, (long)qt * BT, &a0, &a1);
            // local + global: the window interval plus the tile's global rows, as bits (none for a
            // padding key)
            uint2 bw = (LG && !full) ? lg_half_bits(a0, a1, p.gbits + 4 * qt, wg) : make_uint2(0u, 0u);
            if (j >= p.S) bw = make_uint2(0u, 0u);
            constexpr int MKP = LG ? MK_BITS : MK_INTERVAL;  // the mask form of the tiles that are not FULL
            const uint32_t vec = s_vec + st * 1024;  // -LSE log2 e of the tile's 128 query rows, then -D
            // ALiBi: the slope of this iteration's query head; |i - j| = |c - (j - first row of the tile)|
            const float mL = AL ? p.alibi[iter_head(it) - b * p.Hq] * LOG2E : 0.f;
            const float base = (float)(j - (long)qt * BT);
            wait_bounded(bar(KV_QFULL + st), (it >> 1) & 1, wd, ERR_COMPUTE);  // the column vectors
            wait_bounded(bar(KV_SFULL), it & 1, wd, ERR_COMPUTE);
            tc_fence_after();
            if constexpr (BM) {  // the bias column of this key over the warpgroup's 64 query rows
                const int a_it = iter_head(it) - b * p.Hq;
                const size_t plane = (size_t)(p.bias_Bb == 1 ? 0 : b) * p.bias_Hb + (p.bias_Hb == 1 ? 0 : a_it);
                const long r0 = (long)qt * BT + wg * HALF;
                const ColBias cbias{j < p.S ? p.bias + (plane * (size_t)p.S + (size_t)r0) * (size_t)p.bias_ld + j : nullptr,
                                    p.bias_ld, (int)min((long)HALF, (long)p.S - r0)};
                if (!full)
                    exp_pass<MKP, true, AL>(t_s, wg, sl2, ColVec{vec}, a0, a1, bw, mL, base, pv, cbias);
                else
                    exp_pass<MK_NONE, true, AL>(t_s, wg, sl2, ColVec{vec}, a0, a1, bw, mL, base, pv, cbias);
            } else {
                if (!full)
                    exp_pass<MKP, true, AL>(t_s, wg, sl2, ColVec{vec}, a0, a1, bw, mL, base, pv);
                else
                    exp_pass<MK_NONE, true, AL>(t_s, wg, sl2, ColVec{vec}, a0, a1, bw, mL, base, pv);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(KV_PDONE + wg));
            wait_bounded(bar(KV_DPFULL), it & 1, wd, ERR_COMPUTE);
            tc_fence_after();
            ds_pass(t_dp, wg, ColVec{vec + 4 * BT}, pv);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(KV_HDONE + wg));
        }
        // epilogue: warpgroup 0 stages dV in the first Q stage, warpgroup 1 stages scale * dK in
        // the first dO stage (both idle once every product has completed), then TMA stores
        wait_bounded(bar(KV_DONE), 0, wd, ERR_COMPUTE);
        tc_fence_after();
        if (wg == 0) stage_groups<D / 32>(smem + C::OFF_Q, t_lane, C::TMEM_DV, 0, t, 1.f);
        else stage_groups<D / 32>(smem + C::OFF_DO, t_lane, C::TMEM_DK, 0, t, p.scale);
        fence_proxy_async_smem();
        named_bar_sync(1, NCOMPUTE);
        if (threadIdx.x == 0 && !sh->abort) {
            for (int s = 0; s < D / 64; ++s) {
                tma_store_3d(&p.tm_dv, s_q + s * C::SUB, s * 64, kv_tile * BT, bkv);
                tma_store_3d(&p.tm_dk, s_do + s * C::SUB, s * 64, kv_tile * BT, bkv);
            }
            tma_store_commit_and_wait_read();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <class F>
cudaError_t configure(F kernel, int smem) {
    return smem_opt_in(reinterpret_cast<const void*>(kernel), smem);
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdPrepParams& p, cudaStream_t stream) {
    if (p.d != 64 && p.d != 128) return cudaErrorInvalidValue;
    const long rows = (long)p.BHq * p.S_pad;
    const long per_block = (long)PREP_WARPS * PREP_ROUNDS * (32 / (p.d / 8));
    bwd_prep_kernel<<<(unsigned)((rows + per_block - 1) / per_block), PREP_WARPS * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D, bool AL, bool BM, bool LG>
cudaError_t launch_dq(const BwdParams& p, int n_items, cudaStream_t stream) {
    cudaError_t e = configure(attn_bwd_dq_kernel<D, AL, BM, LG>, DqCfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attn_bwd_dq_kernel<D, AL, BM, LG><<<n_items, NTHREADS, DqCfg<D>::SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

template <int D, bool AL, bool BM, bool LG>
cudaError_t launch_dkdv(const BwdParams& p, int n_ctas, cudaStream_t stream) {
    cudaError_t e = configure(attn_bwd_dkdv_kernel<D, AL, BM, LG>, KvCfg<D>::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attn_bwd_dkdv_kernel<D, AL, BM, LG><<<n_ctas, NTHREADS, KvCfg<D>::SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

// local + global (p.list set): plain, with ALiBi or with a bias matrix
template <int D>
cudaError_t launch_dq_d(const BwdParams& p, int n_items, cudaStream_t stream) {
    if (p.list) {
        if (p.bias) return launch_dq<D, false, true, true>(p, n_items, stream);
        if (p.alibi) return launch_dq<D, true, false, true>(p, n_items, stream);
        return launch_dq<D, false, false, true>(p, n_items, stream);
    }
    if (p.bias) return launch_dq<D, false, true, false>(p, n_items, stream);
    if (p.alibi) return launch_dq<D, true, false, false>(p, n_items, stream);
    return launch_dq<D, false, false, false>(p, n_items, stream);
}

template <int D>
cudaError_t launch_dkdv_d(const BwdParams& p, int n_ctas, cudaStream_t stream) {
    if (p.list) {
        if (p.bias) return launch_dkdv<D, false, true, true>(p, n_ctas, stream);
        if (p.alibi) return launch_dkdv<D, true, false, true>(p, n_ctas, stream);
        return launch_dkdv<D, false, false, true>(p, n_ctas, stream);
    }
    if (p.bias) return launch_dkdv<D, false, true, false>(p, n_ctas, stream);
    if (p.alibi) return launch_dkdv<D, true, false, false>(p, n_ctas, stream);
    return launch_dkdv<D, false, false, false>(p, n_ctas, stream);
}

cudaError_t launch_bwd_dq(const BwdParams& p, int d, int n_items, cudaStream_t stream) {
    if (n_items <= 0) return cudaSuccess;
    if (d == 128) return launch_dq_d<128>(p, n_items, stream);
    if (d == 64) return launch_dq_d<64>(p, n_items, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, int n_ctas, cudaStream_t stream) {
    if (n_ctas <= 0) return cudaSuccess;
    if (d == 128) return launch_dkdv_d<128>(p, n_ctas, stream);
    if (d == 64) return launch_dkdv_d<64>(p, n_ctas, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
