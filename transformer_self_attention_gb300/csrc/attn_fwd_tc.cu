// Tensor-core attention forward for sm_103a (bf16 in, fp32 accumulation).
//
// One CTA computes one work item: 128 query rows of one (batch, query head)
// against the key tiles the host schedule lists for them.  The pages' design
// (tiling Q into blocks, streaming K/V blocks, keeping a running row max m and
// sum l and writing only O back -- "Transformer 演进与变体" (ai.icyfenix.cn),
// section Flash Attention; the m/l recurrence also in "Trasformer 浅析",
// section 长序列的三条优化路线) is mapped onto Blackwell as follows:
//
//   warp 4 (producer) : TMA loads of the Q tile (once) and of every K and V
//                       tile into 128B-swizzled shared memory.
//   warp 5 (MMA)      : one thread issues tcgen05.mma: S = Q K^T into tensor
//                       memory (fp32), then O += P V with P read from tensor
//                       memory (bf16) and O accumulated in tensor memory.
//   warps 0-3         : one thread per query row.  Load the row of S from
//                       tensor memory, apply the mask on PARTIAL tiles, update
//                       the running max/sum with exp2 on log2(e)-prescaled
//                       scores, write P (bf16) back over S, and rescale the O
//                       row only when the running max grew by more than 2^8
//                       (the final division by l keeps the result exact).
//                       P is released in two halves of 64 keys: the MMA thread
//                       starts O += P V on the first half while the second is
//                       still being exponentiated.
//                       Epilogue: O / l -> bf16 -> swizzled smem -> TMA store;
//                       LSE = (m + log2 l) ln 2.
//
// Tensor memory: S/P in columns [0, 128), O in [128, 128 + d); 256 columns per
// CTA, so two CTAs share an SM and one's softmax overlaps the other's MMAs.
//
// Local + global ("Transformer 演进与变体", section 稀疏注意力) runs as one launch of
// its own instantiation (LG):
//   * a query tile's global keys outside its band of key tiles are gathered by the
//     producer warp (plain loads into the swizzled layout) into narrow key tiles of
//     32, 64, 96 or 128 columns (at most the kernel's tile width), every column allowed
//     for every row, taken before the band tiles;
//   * the global rows are computed by their own items against every key, split into key
//     chunks; each chunk writes a partial result and the last chunk of a row tile to
//     finish (an arrival counter) merges them into O and LSE;
//   * band items skip the stores of the global rows their tile holds.
// Every wait on an mbarrier is bounded by a wall-clock limit; a wait that runs
// out records an error bit, raises a CTA-wide abort flag and the CTA drains
// its in-flight copies and MMAs (again bounded), frees tensor memory and exits.
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_once.h"
#include "kernels.h"
#include "sm103_ptx.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;            // query rows per CTA
constexpr int KT = 128;            // keys per tile of the host schedule (a kernel tile is KT or KT / 2 keys)
constexpr int NTHREADS = 192;      // 4 softmax warps + producer + MMA
constexpr int WARP_PRODUCER = 4;
constexpr int WARP_MMA = 5;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units: rescale O only if the max grew by > 2^8

enum : int { ERR_PRODUCER = 1, ERR_MMA = 2, ERR_SOFTMAX = 4 };

// BIAS: 0 none; 1 ALiBi added per element (symmetric kinds, |i - j|); 2 ALiBi under the
// causal kinds, added by the tensor core (see the MMA role); 3 a given bias matrix b_ij.
enum { BIAS_NONE = 0, BIAS_ALIBI_ELEM = 1, BIAS_ALIBI_MMA = 2, BIAS_MATRIX = 3 };

// BN_: keys per kernel tile.  128 everywhere except d = 64 without a score bias, which takes 64-key
// tiles: S (64 columns) and O (64) then fit in 128 tensor-memory columns, so four CTAs -- four
// S -> softmax -> PV chains -- share an SM instead of two.  At d = 64 a 128-key tile carries half the
// products of d = 128 but the same softmax and hand-off latency, and two chains leave the tensor pipe
// idle most of the time.
template <int D, int BIAS = BIAS_NONE, bool F8 = false, int BN_ = 128>
struct Cfg {
    static_assert(BN_ == 128 || (BN_ == 64 && D == 64 && BIAS == BIAS_NONE && !F8), "64-key tiles: d = 64, bf16, no bias");
    static constexpr int BN = BN_;                // keys per kernel tile
    static constexpr int SUBT = KT / BN;          // kernel tiles per schedule tile
    static constexpr int EB = F8 ? 1 : 2;         // bytes per element (E4M3 or bf16)
    static constexpr int ROWB = D * EB;           // bytes per row of Q, K, V
    // swizzle width: 128-byte blocks, or one 64-byte block for 64-byte rows (E4M3 at d = 64)
    static constexpr int SWB = ROWB < 128 ? ROWB : 128;
    static_assert(SWB == 128 || SWB == 64, "row layout");
    static constexpr uint32_t SW_MODE = SWB == 128 ? 2u : 4u;  // shared-memory descriptor swizzle field
    static constexpr int SBO = 8 * SWB;           // descriptor stride between 8-row groups
    static constexpr int SPB = SWB / 32;          // 32-byte K steps per block row
    static constexpr int SUB = BM * SWB;          // bytes of one 128-row swizzled block of Q
    static constexpr int KV_SUB = BN * SWB;       // the same for a K / V tile of BN rows
    static constexpr int OSUB = BM * 128;         // one 64-column block of the bf16 O staging
    static constexpr int XW = SWB / EB;           // elements per row of a block
    static constexpr int NSUB = ROWB / SWB;       // blocks per row
    static constexpr int TILE_BYTES = BM * ROWB;  // one Q tile
    static constexpr int KV_BYTES = BN * ROWB;    // one K / V tile
    // rows of the K / V tensor maps' box (the host encodes 64 at d = 64, 128 otherwise); a tile of BN
    // rows is BN / KV_BOX copies per 64-column block
    static constexpr int KV_BOX = (D == 64) ? 64 : 128;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + TILE_BYTES;
    static constexpr int OFF_V = OFF_K + KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + KV_BYTES;
    // BIAS_ALIBI_MMA: a ones block and a bias block, each 128 rows x 16 bf16 (K-major, no swizzle)
    static constexpr int OFF_BA = OFF_BAR + 1024;
    static constexpr int OFF_BB = OFF_BA + 4096;
    static constexpr int SMEM_USED = (BIAS == BIAS_ALIBI_MMA) ? OFF_BB + 4096 : OFF_BAR + 128;
    // CTAs per SM: as many as tensor memory holds (two of 256 columns, or four of 128); the shared
    // memory request keeps the count from going higher (a CTA beyond them would wait for its columns)
    static constexpr int CTAS_PER_SM = (BN == 64) ? 4 : 2;
    static constexpr int SMEM_MIN = (BN == 64) ? 46 * 1024 : 82 * 1024;
    static constexpr int SMEM_ALLOC = (SMEM_USED + 1024 > SMEM_MIN) ? SMEM_USED + 1024 : SMEM_MIN;
    static constexpr uint32_t TMEM_COLS = (BN == 64) ? 128 : 256;
    static constexpr uint32_t TMEM_S = 0;
    static constexpr uint32_t TMEM_O = BN;
};

// B_PFULL / B_PFULL1: the first / second half of P (keys 0-63 / 64-127) is in tensor memory.
enum Bar { B_Q = 0, B_KFULL, B_KEMPTY, B_VFULL, B_VEMPTY, B_SFULL, B_PFULL, B_PFULL1, B_OFULL, NBAR };

struct Shared {  // small control block after the tiles
    uint64_t bar[NBAR];
    uint32_t tmem_base;
    volatile int abort;
    volatile int merge_last; // global-row chunk items: this CTA finished last and merges the chunks
};

// Bounded wait: polls the barrier; every 128 polls checks the CTA abort flag
// and the wall clock.  Returns false (after raising the abort flag and the
// error bit) if the limit ran out or another role aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Shared* sh, const TcParams& p,
                                             int role) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 127u) == 0) {
            if (sh->abort) return false;
            if ((long long)(globaltimer() - t0) > p.watchdog_ns) {
                sh->abort = 1;
                atomicOr(p.err, role);
                return false;
            }
        }
    }
}

// Drain wait used after an abort: no abort check, only the clock.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const TcParams& p) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if ((long long)(globaltimer() - t0) > p.watchdog_ns) return;
}

// Bounded busy wait on the non-blocking test (lowest wake-up latency; for the
// single MMA-issuing thread, which has nothing else to do meanwhile).
__device__ __forceinline__ bool spin_bounded(uint32_t bar, uint32_t parity, Shared* sh, const TcParams& p, int role) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((n & 1023u) == 0) {
            if (sh->abort) return false;
            if ((long long)(globaltimer() - t0) > p.watchdog_ns) {
                sh->abort = 1;
                atomicOr(p.err, role);
                return false;
            }
        }
    }
}

// Mask of one PARTIAL tile as seen by one query row: the allowed in-tile columns are
// [a0, a1] (clamped to [-1, tile width]) plus the global keys of the tile.  w0..w3 hold them as
// one bit per column (filled for the MASK_ANY form only), so that testing a column is one
// bit test and one select.
struct TileMask {
    int a0, a1;
    uint32_t w0, w1, w2, w3;
};

// Bits of the columns [32k, 32k + 32) that lie inside [a0, a1].
__device__ __forceinline__ uint32_t interval_word(int a0, int a1, int k) {
    const int lo = max(a0 - 32 * k, 0), hi = min(a1 - 32 * k + 1, 32);  // [lo, hi)
    if (hi <= lo) return 0u;
    const uint32_t up = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
    return up & ~((1u << lo) - 1u);
}

__device__ __forceinline__ bool tile_allowed(int c, const TileMask& mk) {
    const uint32_t w = c < 32 ? mk.w0 : c < 64 ? mk.w1 : c < 96 ? mk.w2 : mk.w3;
    return (w >> (c & 31)) & 1u;
}

// Mask forms of a tile, decided once per tile and warp-uniformly:
//   MASK_NONE  : FULL tile, no predicate;
//   MASK_UPPER : allowed columns are c <= a1 (a0 <= 0, no global keys) -- the causal diagonal
//                tiles; one compare and one select per element;
//   MASK_ANY   : the interval [a0, a1] plus the global keys, as the column bits w0..w3.
enum { MASK_NONE = 0, MASK_UPPER = 1, MASK_ANY = 2 };

template <int MASKED>
__device__ __forceinline__ float tile_score(uint32_t raw, int c, const TileMask& mk) {
    if (MASKED == MASK_NONE) return __uint_as_float(raw);
    if (MASKED == MASK_UPPER) return c <= mk.a1 ? __uint_as_float(raw) : -INFINITY;
    return tile_allowed(c, mk) ? __uint_as_float(raw) : -INFINITY;
}

// Row maximum of the (masked) raw scores of this thread's row, columns [0, NB):
// three-input max instructions, eight independent chains.
template <int MASKED, int NB = 128>
__device__ __forceinline__ float tile_row_max(uint32_t t_s, const TileMask& mk) {
    float m8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
    for (int h = 0; h < NB / 64; ++h) {
        uint32_t r0[32], r1[32];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const int k = (e >> 1) & 7;
            m8[k] = fmax3(m8[k], tile_score<MASKED>(r0[e], h * 64 + e, mk), tile_score<MASKED>(r0[e + 1], h * 64 + e + 1, mk));
            m8[k] = fmax3(m8[k], tile_score<MASKED>(r1[e], h * 64 + 32 + e, mk),
                          tile_score<MASKED>(r1[e + 1], h * 64 + 33 + e, mk));
        }
    }
    return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// Announce the first half of P (keys 0-63) to the MMA thread once this thread's stores of it
// have landed; the thread's O rescale, if any, came before.
__device__ __forceinline__ void release_first_half(uint32_t bar_half) {
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(bar_half);
}

// P = exp2(s * sl2 - ref) written as bf16 over the S columns; returns the row sum.
// Half h (keys 64h .. 64h+63) reads S columns [64h, 64h+64) and writes P columns
// [32h, 32h+32), which only overlap S columns this thread has already read.  The
// scale-and-subtract and the running sums use the packed two-lane fp32 instructions.
// The first half is announced on bar_half as soon as it is stored.  fix() (the row's lazy O
// rescale and running-sum update) runs after that half is computed and before it is announced:
// it is off the path from S to the first exponentials, and O is rescaled before O += P V starts.
template <int MASKED, typename FixO>
__device__ __forceinline__ float tile_exp_store(uint32_t t_s, const TileMask& mk, float sl2, float ref,
                                               uint32_t bar_half, FixO&& fix) {
    const float2 sl2x2 = make_float2(sl2, sl2), nref = make_float2(-ref, -ref);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r0[32], r1[32], pk[32];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float2 x01 = __ffma2_rn(make_float2(tile_score<MASKED>(r0[2 * e], h * 64 + 2 * e, mk),
                                                      tile_score<MASKED>(r0[2 * e + 1], h * 64 + 2 * e + 1, mk)),
                                          sl2x2, nref);
            const float2 x23 = __ffma2_rn(make_float2(tile_score<MASKED>(r1[2 * e], h * 64 + 32 + 2 * e, mk),
                                                      tile_score<MASKED>(r1[2 * e + 1], h * 64 + 33 + 2 * e, mk)),
                                          sl2x2, nref);
            const float p0 = ex2(x01.x), p1 = ex2(x01.y), p2 = ex2(x23.x), p3 = ex2(x23.y);
            acc0 = __fadd2_rn(acc0, make_float2(p0, p1));
            acc1 = __fadd2_rn(acc1, make_float2(p2, p3));
            pk[e] = pack_bf16x2(p0, p1);
            pk[16 + e] = pack_bf16x2(p2, p3);
        }
        tmem_st32(t_s + h * 32, pk);
        if (h == 0) {
            fix();
            release_first_half(bar_half);
        }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// tile_exp_store for 64-key tiles: halves of 32 keys (S columns [32h, 32h + 32) in, bf16 P columns
// [16h, 16h + 16) out, again only over S columns already read), the first half announced on
// bar_half after fix().
template <int MASKED, typename FixO>
__device__ __forceinline__ float tile_exp_store_n64(uint32_t t_s, const TileMask& mk, float sl2, float ref,
                                                   uint32_t bar_half, FixO&& fix) {
    const float2 sl2x2 = make_float2(sl2, sl2), nref = make_float2(-ref, -ref);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r[32], pk[16];
        tmem_ld32(t_s + h * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = h * 32 + 4 * e;
            const float2 x01 = __ffma2_rn(make_float2(tile_score<MASKED>(r[4 * e], c, mk),
                                                      tile_score<MASKED>(r[4 * e + 1], c + 1, mk)),
                                          sl2x2, nref);
            const float2 x23 = __ffma2_rn(make_float2(tile_score<MASKED>(r[4 * e + 2], c + 2, mk),
                                                      tile_score<MASKED>(r[4 * e + 3], c + 3, mk)),
                                          sl2x2, nref);
            const float p0 = ex2(x01.x), p1 = ex2(x01.y), p2 = ex2(x23.x), p3 = ex2(x23.y);
            acc0 = __fadd2_rn(acc0, make_float2(p0, p1));
            acc1 = __fadd2_rn(acc1, make_float2(p2, p3));
            pk[2 * e] = pack_bf16x2(p0, p1);
            pk[2 * e + 1] = pack_bf16x2(p2, p3);
        }
        tmem_st16(t_s + h * 16, pk);
        if (h == 0) {
            fix();
            release_first_half(bar_half);
        }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// tile_exp_store for E4M3 P: four keys per 32-bit tensor-memory column (the A operand
// layout of the 8-bit MMA), keys 4q..4q+3 of half h in column 16h + q.  P <= 2^8 by the
// lazy rescale, inside the E4M3 range (448).
template <int MASKED>
__device__ __forceinline__ float tile_exp_store_e4m3(uint32_t t_s, const TileMask& mk, float sl2, float ref,
                                                    uint32_t bar_half) {
    const float2 sl2x2 = make_float2(sl2, sl2), nref = make_float2(-ref, -ref);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r0[32], r1[32], pk[16];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float pa[4], pb[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
                const int c0 = h * 64 + 4 * q + u, c1 = h * 64 + 32 + 4 * q + u;
                const float2 xa = __ffma2_rn(make_float2(tile_score<MASKED>(r0[4 * q + u], c0, mk),
                                                         tile_score<MASKED>(r0[4 * q + u + 1], c0 + 1, mk)), sl2x2, nref);
                const float2 xb = __ffma2_rn(make_float2(tile_score<MASKED>(r1[4 * q + u], c1, mk),
                                                         tile_score<MASKED>(r1[4 * q + u + 1], c1 + 1, mk)), sl2x2, nref);
                pa[u] = ex2(xa.x); pa[u + 1] = ex2(xa.y);
                pb[u] = ex2(xb.x); pb[u + 1] = ex2(xb.y);
                acc0 = __fadd2_rn(acc0, make_float2(pa[u], pa[u + 1]));
                acc1 = __fadd2_rn(acc1, make_float2(pb[u], pb[u + 1]));
            }
            pk[q] = pack_e4m3x4(pa[0], pa[1], pa[2], pa[3]);
            pk[8 + q] = pack_e4m3x4(pb[0], pb[1], pb[2], pb[3]);
        }
        tmem_st16(t_s + h * 16, pk);
        if (h == 0) release_first_half(bar_half);
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// The same two passes with the additive bias -m_a |i - j| of ALiBi, in log2 units:
// x = s * sl2 - mL * |base - c| for in-tile column c, with mL = m_a log2(e) and
// base = i - (first key of the tile).  Under the causal kinds every allowed key has
// j <= i, so |base - c| = base - c and the bias is linear in c (ABS = false); the
// symmetric kinds take the absolute value.  Masked scores are -inf and stay -inf.
template <bool ABS>
__device__ __forceinline__ float2 alibi_pair(float base, int c, float mL, float sub) {
    // -mL * |base - c| - sub and -mL * |base - c - 1| - sub
    if constexpr (ABS)
        return make_float2(fmaf(-mL, fabsf(base - (float)c), -sub), fmaf(-mL, fabsf(base - (float)(c + 1)), -sub));
    else
        return __ffma2_rn(make_float2((float)c, (float)(c + 1)), make_float2(mL, mL),
                          make_float2(fmaf(-mL, base, -sub), fmaf(-mL, base, -sub)));
}

// Row maximum of x (log2 units, no further scaling).
template <int MASKED, bool ABS>
__device__ __forceinline__ float tile_row_max_alibi(uint32_t t_s, const TileMask& mk, float sl2, float mL,
                                                    float base) {
    const float2 sl2x2 = make_float2(sl2, sl2);
    float m8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r0[32], r1[32];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const int c0 = h * 64 + e, c1 = h * 64 + 32 + e;
            const float2 x0 = __ffma2_rn(make_float2(tile_score<MASKED>(r0[e], c0, mk), tile_score<MASKED>(r0[e + 1], c0 + 1, mk)),
                                         sl2x2, alibi_pair<ABS>(base, c0, mL, 0.f));
            const float2 x1 = __ffma2_rn(make_float2(tile_score<MASKED>(r1[e], c1, mk), tile_score<MASKED>(r1[e + 1], c1 + 1, mk)),
                                         sl2x2, alibi_pair<ABS>(base, c1, mL, 0.f));
            const int k = (e >> 1) & 7;
            m8[k] = fmax3(m8[k], x0.x, x0.y);
            m8[k] = fmax3(m8[k], x1.x, x1.y);
        }
    }
    return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

template <int MASKED, bool ABS>
__device__ __forceinline__ float tile_exp_store_alibi(uint32_t t_s, const TileMask& mk, float sl2, float ref,
                                                      float mL, float base, uint32_t bar_half) {
    const float2 sl2x2 = make_float2(sl2, sl2);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r0[32], r1[32], pk[32];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int c0 = h * 64 + 2 * e, c1 = h * 64 + 32 + 2 * e;
            const float2 x01 = __ffma2_rn(make_float2(tile_score<MASKED>(r0[2 * e], c0, mk), tile_score<MASKED>(r0[2 * e + 1], c0 + 1, mk)),
                                          sl2x2, alibi_pair<ABS>(base, c0, mL, ref));
            const float2 x23 = __ffma2_rn(make_float2(tile_score<MASKED>(r1[2 * e], c1, mk), tile_score<MASKED>(r1[2 * e + 1], c1 + 1, mk)),
                                          sl2x2, alibi_pair<ABS>(base, c1, mL, ref));
            const float p0 = ex2(x01.x), p1 = ex2(x01.y), p2 = ex2(x23.x), p3 = ex2(x23.y);
            acc0 = __fadd2_rn(acc0, make_float2(p0, p1));
            acc1 = __fadd2_rn(acc1, make_float2(p2, p3));
            pk[e] = pack_bf16x2(p0, p1);
            pk[16 + e] = pack_bf16x2(p2, p3);
        }
        tmem_st32(t_s + h * 32, pk);
        if (h == 0) release_first_half(bar_half);
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// tile_exp_store_alibi for E4M3 P (four keys per tensor-memory column, as tile_exp_store_e4m3).
template <int MASKED, bool ABS>
__device__ __forceinline__ float tile_exp_store_alibi_e4m3(uint32_t t_s, const TileMask& mk, float sl2, float ref,
                                                           float mL, float base, uint32_t bar_half) {
    const float2 sl2x2 = make_float2(sl2, sl2);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r0[32], r1[32], pk[16];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float pa[4], pb[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
                const int c0 = h * 64 + 4 * q + u, c1 = h * 64 + 32 + 4 * q + u;
                const float2 xa = __ffma2_rn(make_float2(tile_score<MASKED>(r0[4 * q + u], c0, mk),
                                                         tile_score<MASKED>(r0[4 * q + u + 1], c0 + 1, mk)),
                                             sl2x2, alibi_pair<ABS>(base, c0, mL, ref));
                const float2 xb = __ffma2_rn(make_float2(tile_score<MASKED>(r1[4 * q + u], c1, mk),
                                                         tile_score<MASKED>(r1[4 * q + u + 1], c1 + 1, mk)),
                                             sl2x2, alibi_pair<ABS>(base, c1, mL, ref));
                pa[u] = ex2(xa.x); pa[u + 1] = ex2(xa.y);
                pb[u] = ex2(xb.x); pb[u + 1] = ex2(xb.y);
                acc0 = __fadd2_rn(acc0, make_float2(pa[u], pa[u + 1]));
                acc1 = __fadd2_rn(acc1, make_float2(pb[u], pb[u + 1]));
            }
            pk[q] = pack_e4m3x4(pa[0], pa[1], pa[2], pa[3]);
            pk[8 + q] = pack_e4m3x4(pb[0], pb[1], pb[2], pb[3]);
        }
        tmem_st16(t_s + h * 16, pk);
        if (h == 0) release_first_half(bar_half);
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// The bias row of this thread for one key tile: 16 loads of 16 bytes (8 keys each), issued
// before the wait for S so that their latency hides behind it.  brow: the row's bias at the
// tile's first key (16-byte aligned), or null for rows past the sequence; chunks of 8 keys are
// read only while they start inside [0, n_valid) (the row stride is a multiple of 8, so a chunk
// that starts there stays inside the row).
__device__ __forceinline__ void load_bias_row(uint4 (&bv)[16], const uint16_t* brow, int n_valid) {
#pragma unroll
    for (int q = 0; q < 16; ++q)
        bv[q] = (brow != nullptr && q * 8 < n_valid) ? __ldg(reinterpret_cast<const uint4*>(brow + q * 8))
                                                   : make_uint4(0, 0, 0, 0);
}

// Pass 1 with a bias matrix: x = s * sl2 + b_ij log2(e), -inf where masked (the mask is applied
// after the add, so padding values of the bias rows never matter), written back over the S
// columns as fp32 -- pass 2 then reads x with unit scale and no mask.  Returns the row max of x.
template <int MASKED>
__device__ __forceinline__ float tile_row_max_matbias(uint32_t t_s, const TileMask& mk, float sl2,
                                                      const uint4 (&bv)[16]) {
    constexpr float LOG2E_F = 1.4426950408889634f;
    const float2 sl2x2 = make_float2(sl2, sl2), l2x2 = make_float2(LOG2E_F, LOG2E_F);
    float m4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) m4[k] = -INFINITY;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {  // 32 keys at a time
        uint32_t r[32];
        tmem_ld32(t_s + ch * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const int c = ch * 32 + e;
            const uint4 w4 = bv[c >> 3];
            const int wi = (e >> 1) & 3;
            const uint32_t w = wi == 0 ? w4.x : wi == 1 ? w4.y : wi == 2 ? w4.z : w4.w;
            const float2 bb = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
            float2 x = __ffma2_rn(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sl2x2,
                                  __fmul2_rn(bb, l2x2));
            if (MASKED) {
                x.x = tile_allowed(c, mk) ? x.x : -INFINITY;
                x.y = tile_allowed(c + 1, mk) ? x.y : -INFINITY;
            }
            r[e] = __float_as_uint(x.x);
            r[e + 1] = __float_as_uint(x.y);
            const int k = (e >> 1) & 3;
            m4[k] = fmax3(m4[k], x.x, x.y);
        }
        tmem_st32(t_s + ch * 32, r);
    }
    tmem_wait_st();
    return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// Rows pos(r), r < n_rows, of one head of ROWB-byte rows (d bf16 or E4M3 values) copied with plain
// loads into a tile of `rows` rows in the layout the TMA loads write.  128-byte swizzle (rows of 128
// bytes or more): blocks of rows * 128 bytes, one per 128 bytes of a row, the 16-byte chunk c of row r
// at chunk position c ^ (r & 7).  64-byte swizzle (64-byte rows): the chunk c (of 4) of row r at
// position c ^ ((r >> 1) & 3).  pos(r) < 0 gives a zero row.  All 32 lanes of one warp take part.
template <int ROWB, class Pos>
__device__ __forceinline__ void gather_rows(uint8_t* tile, int rows, const void* head, int n_rows, Pos pos,
                                            int lane) {
    constexpr int CH = ROWB / 16;  // 16-byte chunks per row
    const uint8_t* h = static_cast<const uint8_t*>(head);
    for (int e = lane; e < n_rows * CH; e += 32) {
        const int r = e / CH, c = e - r * CH;
        const long j = pos(r);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (j >= 0) v = __ldg(reinterpret_cast<const uint4*>(h + j * ROWB) + c);
        if constexpr (ROWB >= 128)
            *reinterpret_cast<uint4*>(tile + (c >> 3) * (rows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        else
            *reinterpret_cast<uint4*>(tile + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) = v;
    }
}

// Row maximum over the first 32 * nch columns of a gathered-key tile (columns > a1 hold no key).
__device__ __forceinline__ float narrow_row_max(uint32_t t_s, int nch, int a1) {
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        uint32_t r[32];
        tmem_ld32(t_s + ch * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const int c = ch * 32 + e;
            m0 = fmax3(m0, c <= a1 ? __uint_as_float(r[e]) : -INFINITY,
                       c + 1 <= a1 ? __uint_as_float(r[e + 1]) : -INFINITY);
            m1 = fmax3(m1, c + 2 <= a1 ? __uint_as_float(r[e + 2]) : -INFINITY,
                       c + 3 <= a1 ? __uint_as_float(r[e + 3]) : -INFINITY);
        }
    }
    return fmaxf(m0, m1);
}

// P = exp2(s * sl2 - ref) over the first 32 * nch columns of a gathered-key tile, bf16 P written
// over S (keys 32ch .. 32ch + 31 in columns 16ch .. 16ch + 15); returns the row sum.  fix() runs
// once every exponential is computed, then the whole of P is announced on bar_p.
template <typename FixO>
__device__ __forceinline__ float narrow_exp_store(uint32_t t_s, int nch, int a1, float sl2, float ref,
                                                  uint32_t bar_p, FixO&& fix) {
    const float2 sl2x2 = make_float2(sl2, sl2), nref = make_float2(-ref, -ref);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        uint32_t r[32], pk[16];
        tmem_ld32(t_s + ch * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int c = ch * 32 + 2 * e;
            const float2 x = __ffma2_rn(make_float2(c <= a1 ? __uint_as_float(r[2 * e]) : -INFINITY,
                                                    c + 1 <= a1 ? __uint_as_float(r[2 * e + 1]) : -INFINITY),
                                        sl2x2, nref);
            const float p0 = ex2(x.x), p1 = ex2(x.y);
            acc = __fadd2_rn(acc, make_float2(p0, p1));
            pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + ch * 16, pk);
    }
    fix();
    release_first_half(bar_p);
    return acc.x + acc.y;
}

// narrow_exp_store for E4M3 P: 64 keys at a time (the columns past 32 * nch hold no key and are
// masked), four keys per tensor-memory column in the A operand layout of the 8-bit MMA (keys
// 4q .. 4q + 3 of a 64-key group h in column 16h + q).  fix() runs once every exponential is
// computed, then the whole of P is announced on bar_p.
template <typename FixO>
__device__ __forceinline__ float narrow_exp_store_e4m3(uint32_t t_s, int nch, int a1, float sl2, float ref,
                                                       uint32_t bar_p, FixO&& fix) {
    float acc = 0.f;
#pragma unroll 1
    for (int h = 0; 2 * h < nch; ++h) {
        uint32_t r0[32], r1[32], pk[16];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float pa[4], pb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int ca = h * 64 + 4 * q + u, cb = ca + 32;
                pa[u] = ex2(ca <= a1 ? fmaf(__uint_as_float(r0[4 * q + u]), sl2, -ref) : -INFINITY);
                pb[u] = ex2(cb <= a1 ? fmaf(__uint_as_float(r1[4 * q + u]), sl2, -ref) : -INFINITY);
                acc += pa[u] + pb[u];
            }
            pk[q] = pack_e4m3x4(pa[0], pa[1], pa[2], pa[3]);
            pk[8 + q] = pack_e4m3x4(pb[0], pb[1], pb[2], pb[3]);
        }
        tmem_st16(t_s + h * 16, pk);
    }
    fix();
    release_first_half(bar_p);
    return acc;
}

// The two passes over a gathered-key tile with the ALiBi bias: x = s sl2 - mL |fi - pos(c)| in log2 units,
// with pos(c) the sequence position of the key in column c and fi the row's; -inf past the tile's keys.
template <class Pos>
__device__ __forceinline__ float narrow_row_max_alibi(uint32_t t_s, int nch, int a1, float sl2, float mL, float fi,
                                                      Pos pos) {
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        uint32_t r[32];
        tmem_ld32(t_s + ch * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const int c = ch * 32 + e;
            const float x0 = c <= a1 ? fmaf(__uint_as_float(r[e]), sl2, -mL * fabsf(fi - pos(c))) : -INFINITY;
            const float x1 = c + 1 <= a1 ? fmaf(__uint_as_float(r[e + 1]), sl2, -mL * fabsf(fi - pos(c + 1))) : -INFINITY;
            m0 = fmaxf(m0, x0);
            m1 = fmaxf(m1, x1);
        }
    }
    return fmaxf(m0, m1);
}

template <class Pos>
__device__ __forceinline__ float narrow_exp_store_alibi(uint32_t t_s, int nch, int a1, float sl2, float ref, float mL,
                                                        float fi, Pos pos, uint32_t bar_p) {
    float acc = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        uint32_t r[32], pk[16];
        tmem_ld32(t_s + ch * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int c = ch * 32 + 2 * e;
            const float x0 = c <= a1 ? fmaf(__uint_as_float(r[2 * e]), sl2, -mL * fabsf(fi - pos(c)) - ref) : -INFINITY;
            const float x1 =
                c + 1 <= a1 ? fmaf(__uint_as_float(r[2 * e + 1]), sl2, -mL * fabsf(fi - pos(c + 1)) - ref) : -INFINITY;
            const float p0 = ex2(x0), p1 = ex2(x1);
            acc += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + ch * 16, pk);
    }
    release_first_half(bar_p);
    return acc;
}

// narrow_exp_store_alibi for E4M3 P: 64 keys at a time, four per tensor-memory column.
template <class Pos>
__device__ __forceinline__ float narrow_exp_store_alibi_e4m3(uint32_t t_s, int nch, int a1, float sl2, float ref,
                                                             float mL, float fi, Pos pos, uint32_t bar_p) {
    float acc = 0.f;
#pragma unroll 1
    for (int h = 0; 2 * h < nch; ++h) {
        uint32_t r0[32], r1[32], pk[16];
        tmem_ld32(t_s + h * 64, r0);
        tmem_ld32(t_s + h * 64 + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float pa[4], pb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int ca = h * 64 + 4 * q + u, cb = ca + 32;
                pa[u] = ex2(ca <= a1 ? fmaf(__uint_as_float(r0[4 * q + u]), sl2, -mL * fabsf(fi - pos(ca)) - ref)
                                     : -INFINITY);
                pb[u] = ex2(cb <= a1 ? fmaf(__uint_as_float(r1[4 * q + u]), sl2, -mL * fabsf(fi - pos(cb)) - ref)
                                     : -INFINITY);
                acc += pa[u] + pb[u];
            }
            pk[q] = pack_e4m3x4(pa[0], pa[1], pa[2], pa[3]);
            pk[8 + q] = pack_e4m3x4(pb[0], pb[1], pb[2], pb[3]);
        }
        tmem_st16(t_s + h * 16, pk);
    }
    release_first_half(bar_p);
    return acc;
}

// Pass 1 over a gathered-key tile with a bias matrix: x = s sl2 + b(i, pos(c)) log2(e) for the
// first 32 * nch columns (-inf past the tile's keys, c > a1), written back over S as fp32 for
// narrow_exp_store with unit scale.  brow: this row's bias (position 0), or null for rows past the
// sequence (their bias reads as 0); pos(c): the key position of column c.  One 2-byte load per key.
template <class Pos>
__device__ __forceinline__ float narrow_row_max_matbias(uint32_t t_s, int nch, int a1, float sl2,
                                                        const uint16_t* brow, Pos pos) {
    constexpr float LOG2E_F = 1.4426950408889634f;
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        uint32_t r[32];
        tmem_ld32(t_s + ch * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const int c = ch * 32 + e;
            const float b0 = (brow && c <= a1) ? __uint_as_float((uint32_t)__ldg(brow + pos(c)) << 16) : 0.f;
            const float b1 = (brow && c + 1 <= a1) ? __uint_as_float((uint32_t)__ldg(brow + pos(c + 1)) << 16) : 0.f;
            const float x0 = c <= a1 ? fmaf(__uint_as_float(r[e]), sl2, b0 * LOG2E_F) : -INFINITY;
            const float x1 = c + 1 <= a1 ? fmaf(__uint_as_float(r[e + 1]), sl2, b1 * LOG2E_F) : -INFINITY;
            r[e] = __float_as_uint(x0);
            r[e + 1] = __float_as_uint(x1);
            m0 = fmaxf(m0, x0);
            m1 = fmaxf(m1, x1);
        }
        tmem_st32(t_s + ch * 32, r);
    }
    tmem_wait_st();
    return fmaxf(m0, m1);
}

// This thread's O row (tensor memory, fp32) times inv_l, stored as bf16 at dst.  Every lane runs
// the tensor-memory loads (they are warp-collective); only lanes with `store` write.
template <int D>
__device__ __forceinline__ void store_row_direct(uint32_t t_o, void* dst_row, float inv_l, bool store) {
    uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + c * 32, o);
        tmem_wait_ld();
        if (store) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(o[8 * q + 2 * e]) * inv_l,
                                        __uint_as_float(o[8 * q + 2 * e + 1]) * inv_l);
                dst[c * 4 + q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
    }
}

// One global row from its key chunks, merged by one warp.  Chunk c holds O_c (its own
// softmax-weighted average, fp32) and LSE_c (natural log of its sum of exponentials), so with
// M = max_c LSE_c the row is
//   O = sum_c e^(LSE_c - M) O_c / sum_c e^(LSE_c - M),   LSE = M + ln sum_c e^(LSE_c - M):
// the softmax normalisation carried across chunks.  The lanes split the chunks for M and the
// weights, then the columns (D / 32 each) for the weighted sum, with four chunks' loads in
// flight.  The partials were written by other CTAs, so they are read through L2 (ld.global.cg).
template <int D>
__device__ __forceinline__ void merge_global_row(const TcParams& p, size_t slot0, void* dst_row, float* lse_out,
                                                 int lane) {
    constexpr int CPL = D / 32;  // columns per lane
    float M = -INFINITY;
    for (int c = lane; c < p.n_chunks; c += 32) M = fmaxf(M, __ldcg(p.part_lse + slot0 + c));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = 0.f;
    float W = 0.f;
    for (int c0 = 0; c0 < p.n_chunks; c0 += 32) {
        const int nc = min(32, p.n_chunks - c0);
        // lane k holds the weight of chunk c0 + k
        const float wl = lane < nc ? expf(__ldcg(p.part_lse + slot0 + c0 + lane) - M) : 0.f;
        W += wl;
#pragma unroll 4
        for (int k = 0; k < nc; ++k) {
            const float w = __shfl_sync(0xffffffffu, wl, k);
            const float* src = p.part_o + (slot0 + c0 + k) * D + lane * CPL;
            if constexpr (CPL == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
                acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
                acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
            } else {
                const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
                acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    const float inv_w = W > 0.f ? 1.f / W : 0.f;
    if constexpr (CPL == 4) {
        reinterpret_cast<uint2*>(dst_row)[lane] =
            make_uint2(pack_bf16x2(acc[0] * inv_w, acc[1] * inv_w), pack_bf16x2(acc[2] * inv_w, acc[3] * inv_w));
    } else {
        reinterpret_cast<uint32_t*>(dst_row)[lane] = pack_bf16x2(acc[0] * inv_w, acc[1] * inv_w);
    }
    if (lse_out && lane == 0) *lse_out = W > 0.f ? M + logf(W) : -INFINITY;
}

template <int D, int BIAS, bool F8, bool LG, int BN>
__global__ void __launch_bounds__(NTHREADS, (Cfg<D, BIAS, F8, BN>::CTAS_PER_SM))
    attn_fwd_tc_kernel(const __grid_constant__ TcParams p) {
    using C = Cfg<D, BIAS, F8, BN>;
    constexpr bool ALIBI = BIAS == BIAS_ALIBI_ELEM;  // the per-element bias passes
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared* sh = reinterpret_cast<Shared*>(smem + C::OFF_BAR);
    const uint32_t s_q = smem_u32(smem + C::OFF_Q);
    const uint32_t s_k = smem_u32(smem + C::OFF_K);
    const uint32_t s_v = smem_u32(smem + C::OFF_V);
    auto bar = [&](int b) { return smem_u32(&sh->bar[b]); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int item = p.item_offset + blockIdx.x;
    const int4 w0 = p.work[2 * item];
    const int4 w1 = p.work[2 * item + 1];
    const int bh = w0.x, q_tile = w0.y, kv_begin = w0.z, kv_end = w0.w;
    const int full_begin = w1.x, full_end = w1.y, flags = w1.z, n_gt = w1.w;
    const bool grows = LG && (flags & ATTN_WORK_GLOBAL_ROWS) != 0;
    // Band key tiles, in kernel tiles of BN keys: the schedule's tiles [kv_begin, kv_end) of KT keys.
    // With 64-key tiles the ends are trimmed to what the rows can see: the query tile's key interval
    // (interval kinds; local + global keeps the schedule's band, outside which its globals are
    // gathered) and, for every item, the sequence end.
    int t_begin = kv_begin * C::SUBT, t_end = kv_end * C::SUBT;
    if constexpr (BN < KT) {
        t_end = min(t_end, (p.S + BN - 1) / BN);
        if (!LG) {
            const long r0 = (long)q_tile * BM, r1 = min(r0 + BM, (long)p.S) - 1;
            long lo0 = 0, hi1 = p.S - 1;
            if (p.kind == ATTN_MASK_CAUSAL) hi1 = r1;
            else if (p.kind == ATTN_MASK_CAUSAL_SLIDING) { lo0 = max(0L, r0 - p.window); hi1 = r1; }
            else if (p.kind == ATTN_MASK_SLIDING) { lo0 = max(0L, r0 - p.window); hi1 = min((long)p.S - 1, r1 + p.window); }
            t_begin = max(t_begin, (int)(lo0 / BN));
            t_end = min(t_end, (int)(hi1 / BN) + 1);
        }
    }
    const int n_band = t_end - t_begin;
    // local + global: the gathered key tiles (n_gat of them, BN keys at most) run before the band tiles,
    // so that the producer warp's plain loads of their rows overlap the copy of the Q tile (measured
    // 3% faster than running them last).  The globals outside the band are G[0, g_lo) and
    // G[g_hi, n_G) (the schedule's split).
    const bool gcols_item = LG && (flags & ATTN_WORK_GLOBAL_COLS);
    const int2 gs = gcols_item ? __ldg(p.gsplit + q_tile) : make_int2(0, p.n_global);
    const int g_lo = gs.x, g_hi = gs.y;
    const int n_out = g_lo + (p.n_global - g_hi);
    const int n_gat = gcols_item ? (n_out + BN - 1) / BN : 0;
    const int n_iter = n_band + n_gat;
    constexpr bool GATHER_FIRST = true;
    auto is_gathered = [&](int it) { return LG && (GATHER_FIRST ? it < n_gat : it >= n_band); };
    auto gat_index = [&](int it) { return GATHER_FIRST ? it : it - n_band; };    // gathered tile of iteration it
    auto band_index = [&](int it) { return GATHER_FIRST ? it - n_gat : it; };   // band position of iteration it
    // Band key tile at band position it.  With the causal ALiBi bias the tiles run from the
    // diagonal downwards: the bias is 0 at j = i and falls with the distance, so a row's running
    // max is set by its first tile and the lazy rescale stays rare.
    constexpr bool REV = BIAS == BIAS_ALIBI_MMA;
    auto band_tile = [&](int it) { return REV ? t_end - 1 - it : t_begin + it; };
    const int b = bh / p.Hq, a = bh - b * p.Hq;
    const int bkv = b * p.Hkv + a / p.group;  // g(a) = a / (Hq / Hkv)

    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i == B_PFULL || i == B_PFULL1) ? 128u : 1u);
        sh->abort = 0;
        sh->merge_last = 0;
        fence_barrier_init();
    }
    if constexpr (BIAS == BIAS_ALIBI_MMA) {
        // Under the causal kinds -m_a |i - j| = -m_a i + m_a (c0 + c) for key c of a tile starting at
        // c0: the softmax of a row ignores the -m_a i and m_a c0 terms until the end (they are folded
        // into the running max and the LSE), and the tensor core adds m_a c / scale to S with one
        // extra K = 16 product: ones [128 x 16] . B^T, B row c = m_a c / scale split into three
        // bf16 terms (hi + mid + lo, about 24 significant bits; the products with one are exact).
        const float sb = p.alibi[a] * 1.4426950408889634f / p.scale_log2;  // m_a / scale
        for (int idx = threadIdx.x; idx < BM * 16; idx += NTHREADS) {
            const int m = idx >> 4, k = idx & 15;
            const uint32_t off = (m >> 3) * 256 + (k >> 3) * 128 + (m & 7) * 16 + (k & 7) * 2;
            const float v = sb * (float)m;
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const float r1 = v - __bfloat162float(hi);
            const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
            const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
            *reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_BA + off) = __float2bfloat16_rn(k < 3 ? 1.f : 0.f);
            *reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_BB + off) =
                k == 0 ? hi : k == 1 ? mid : k == 2 ? lo : __float2bfloat16_rn(0.f);
        }
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
    // gathered key tiles: tile g < n_gat holds the outside keys g * BN .. g * BN + cols(g) - 1,
    // padded to a multiple of 32 columns
    auto gathered_cols = [&](int g) { return min(BN, n_out - g * BN); };
    auto outside_key = [&](int e) -> long { return __ldg(p.globals + (e < g_lo ? e : g_hi + (e - g_lo))); };

    if (LG && warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ producer (local + global)
        // Lane 0 issues the TMA copies and waits for free buffers; all lanes gather the rows of the
        // global tokens (plain loads into the swizzled layout, then a proxy fence so the tensor core
        // sees them, then one arrival).  The gathered key tiles come first, so that their loads
        // overlap the copy of the Q tile.
        if (grows) {  // query rows G[q_tile * BM + r]; rows past the list are zero
            const int r0 = q_tile * BM;
            gather_rows<D * C::EB>(smem + C::OFF_Q, BM, reinterpret_cast<const uint8_t*>(p.q) + (size_t)bh * p.S * D * C::EB, BM,
                           [&](int r) -> long { return r0 + r < p.n_global ? (long)__ldg(p.globals + r0 + r) : -1L; },
                           lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_Q));
        } else if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q), C::TILE_BYTES);
            for (int s = 0; s < C::NSUB; ++s) tma_load_3d(s_q + s * C::SUB, &p.tm_q, bar(B_Q), s * C::XW, q_tile * BM, bh);
        }
        int k_loaded = 0, v_loaded = 0;
        bool ok = true;
        for (int it = 0; it < n_iter && ok; ++it) {
            const bool in_band = !is_gathered(it);
            const int row = in_band ? band_tile(band_index(it)) * BN : 0;
            // gathered tile g: the outside keys g * BN + r, r < ncols, padded with zero rows
            const int gcols = in_band ? 0 : gathered_cols(gat_index(it));
            const int grows_pad = (gcols + 31) & ~31;
            auto gpos = [&](int r) -> long { return r < gcols ? outside_key(gat_index(it) * BN + r) : -1L; };
            if (it > 0) {
                bool w = true;
                if (lane == 0) w = wait_bounded(bar(B_KEMPTY), (it - 1) & 1, sh, p, ERR_PRODUCER);
                if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
            }
            if (in_band) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(B_KFULL), C::KV_BYTES);
                    for (int s = 0; s < C::NSUB; ++s)
                        for (int r = 0; r < BN; r += C::KV_BOX)
                            tma_load_3d(s_k + s * C::KV_SUB + r * C::SWB, &p.tm_k, bar(B_KFULL), s * C::XW, row + r, bkv);
                    if constexpr (BIAS == BIAS_MATRIX)  // the softmax reads this tile's bias rows a tile later
                        if (!grows)
                            tma_prefetch_l2_3d(&p.tm_bias, row, q_tile * BM,
                                               (p.bias_Bb == 1 ? 0 : b) * p.bias_Hb + (p.bias_Hb == 1 ? 0 : a));
                }
            } else {
                gather_rows<D * C::EB>(smem + C::OFF_K, BN, reinterpret_cast<const uint8_t*>(p.k) + (size_t)bkv * p.S * D * C::EB,
                                       grows_pad, gpos, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_KFULL));
            }
            ++k_loaded;
            if (it > 0) {
                bool w = true;
                if (lane == 0) w = wait_bounded(bar(B_VEMPTY), (it - 1) & 1, sh, p, ERR_PRODUCER);
                if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
            }
            if (p.withhold_v) continue;
            if (in_band) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(B_VFULL), C::KV_BYTES);
                    for (int s = 0; s < C::NSUB; ++s)
                        for (int r = 0; r < BN; r += C::KV_BOX)
                            tma_load_3d(s_v + s * C::KV_SUB + r * C::SWB, &p.tm_v, bar(B_VFULL), s * C::XW, row + r, bkv);
                }
            } else {
                gather_rows<D * C::EB>(smem + C::OFF_V, BN, reinterpret_cast<const uint8_t*>(p.v) + (size_t)bkv * p.S * D * C::EB,
                                       grows_pad, gpos, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_VFULL));
            }
            ++v_loaded;
        }
        if (lane == 0 && sh->abort) {  // let the copies this warp issued land before the CTA exits
            drain_wait(bar(B_Q), 0, p);
            if (k_loaded) drain_wait(bar(B_KFULL), (k_loaded - 1) & 1, p);
            if (v_loaded) drain_wait(bar(B_VFULL), (v_loaded - 1) & 1, p);
        }
    } else if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const CUtensorMap* qmap = &p.tm_q;
            const int bias_plane = (BIAS == BIAS_MATRIX)
                                       ? (p.bias_Bb == 1 ? 0 : b) * p.bias_Hb + (p.bias_Hb == 1 ? 0 : a)
                                       : 0;
            if constexpr (BIAS == BIAS_MATRIX) prefetch_tmap(&p.tm_bias);
            mbar_arrive_expect_tx(bar(B_Q), C::TILE_BYTES);
            for (int s = 0; s < C::NSUB; ++s) tma_load_3d(s_q + s * C::SUB, qmap, bar(B_Q), s * C::XW, q_tile * BM, bh);
            int k_loaded = 0, v_loaded = 0;
            bool ok = true;
            for (int it = 0; it < n_iter && ok; ++it) {
                const CUtensorMap* km = &p.tm_k;
                const CUtensorMap* vm = &p.tm_v;
                const int row = band_tile(it) * BN;
                if (it > 0 && !(ok = wait_bounded(bar(B_KEMPTY), (it - 1) & 1, sh, p, ERR_PRODUCER))) break;
                mbar_arrive_expect_tx(bar(B_KFULL), C::KV_BYTES);
                for (int s = 0; s < C::NSUB; ++s)
                    for (int r = 0; r < BN; r += C::KV_BOX)
                        tma_load_3d(s_k + s * C::KV_SUB + r * C::SWB, km, bar(B_KFULL), s * C::XW, row + r, bkv);
                ++k_loaded;
                if constexpr (BIAS == BIAS_MATRIX)  // the softmax reads this tile's bias rows a tile later
                    tma_prefetch_l2_3d(&p.tm_bias, row, q_tile * BM, bias_plane);
                if (it > 0 && !(ok = wait_bounded(bar(B_VEMPTY), (it - 1) & 1, sh, p, ERR_PRODUCER))) break;
                if (p.withhold_v) continue;
                mbar_arrive_expect_tx(bar(B_VFULL), C::KV_BYTES);
                for (int s = 0; s < C::NSUB; ++s)
                    for (int r = 0; r < BN; r += C::KV_BOX)
                        tma_load_3d(s_v + s * C::KV_SUB + r * C::SWB, vm, bar(B_VFULL), s * C::XW, row + r, bkv);
                ++v_loaded;
            }
            if (sh->abort) {  // let the copies this thread issued land before the CTA exits
                drain_wait(bar(B_Q), 0, p);
                if (k_loaded) drain_wait(bar(B_KFULL), (k_loaded - 1) & 1, p);
                if (v_loaded) drain_wait(bar(B_VFULL), (v_loaded - 1) & 1, p);
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = F8 ? idesc_e4m3_f32(BM, BN, false) : idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t idesc_pv = F8 ? idesc_e4m3_f32(BM, D, true) : idesc_bf16_f32(BM, D, true);
            constexpr int KS = F8 ? 32 : 16;  // K elements per MMA (32 bytes of a 128-byte row either way)
            const uint32_t t_s = tmem + C::TMEM_S, t_o = tmem + C::TMEM_O;
            int last_bar = -1, last_par = 0;
            bool ok = wait_bounded(bar(B_Q), 0, sh, p, ERR_MMA);
            for (int it = 0; it < n_iter && ok; ++it) {
                if (!(ok = wait_bounded(bar(B_KFULL), it & 1, sh, p, ERR_MMA))) break;
                // S/P share tensor columns.  No wait for PV(it-1) here: the MMAs one thread issues
                // execute in issue order, so QK(it) overwrites P(it-1) only after PV(it-1) read it.
                tc_fence_after();
                // a gathered-key tile is ncols wide (a multiple of 32): N = ncols for S, K = ncols for P V
                const bool narrow = is_gathered(it);
                const int ncols = narrow ? (gathered_cols(gat_index(it)) + 31) & ~31 : BN;
                const uint32_t idesc_s =
                    narrow ? (F8 ? idesc_e4m3_f32(BM, ncols, false) : idesc_bf16_f32(BM, ncols, false)) : idesc_qk;
#pragma unroll
                for (int k = 0; k < D / KS; ++k) {
                    const uint32_t offq = (k / C::SPB) * C::SUB + (k % C::SPB) * 32,
                                   offk = (k / C::SPB) * C::KV_SUB + (k % C::SPB) * 32;
                    if constexpr (F8)
                        mma_ss_f8(t_s, sdesc_sw(s_q + offq, 16, C::SBO, C::SW_MODE),
                                  sdesc_sw(s_k + offk, 16, C::SBO, C::SW_MODE), idesc_s, k > 0);
                    else
                        mma_ss(t_s, sdesc_sw(s_q + offq, 16, C::SBO, C::SW_MODE),
                               sdesc_sw(s_k + offk, 16, C::SBO, C::SW_MODE), idesc_s, k > 0);
                }
                if constexpr (BIAS == BIAS_ALIBI_MMA)
                    mma_ss(t_s, sdesc_plain(smem_u32(smem + C::OFF_BA), 128, 256),
                           sdesc_plain(smem_u32(smem + C::OFF_BB), 128, 256), idesc_qk, 1u);
                mma_commit(bar(B_SFULL));
                mma_commit(bar(B_KEMPTY));
                last_bar = B_KEMPTY; last_par = it & 1;
                if (!(ok = spin_bounded(bar(B_PFULL), it & 1, sh, p, ERR_MMA))) break;
                // a gathered tile's P is announced whole: wait for both arrivals before its products,
                // so that QK(it+1) is issued only after every softmax thread is done with tile it
                if (narrow && !(ok = spin_bounded(bar(B_PFULL1), it & 1, sh, p, ERR_MMA))) break;
                if (!(ok = wait_bounded(bar(B_VFULL), it & 1, sh, p, ERR_MMA))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / KS; ++k) {
                    if (k * KS >= ncols) break;
                    if (!narrow && k == BN / KS / 2) {  // the second half of P (keys BN/2 .. BN-1)
                        if (!(ok = spin_bounded(bar(B_PFULL1), it & 1, sh, p, ERR_MMA))) break;
                        tc_fence_after();
                    }
                    // P: KS keys = 8 tensor-memory columns (2 bf16 or 4 E4M3 per column);
                    // V: KS key rows of 128 B each (MN-major: d runs along the row)
                    if constexpr (F8)
                        mma_ts_f8(t_o, t_s + k * 8, sdesc_sw(s_v + k * KS * C::SWB, C::KV_SUB, C::SBO, C::SW_MODE), idesc_pv,
                                  (it > 0 || k > 0) ? 1u : 0u);
                    else
                        mma_ts(t_o, t_s + k * 8, sdesc_sw(s_v + k * KS * C::SWB, C::KV_SUB, C::SBO, C::SW_MODE), idesc_pv,
                               (it > 0 || k > 0) ? 1u : 0u);
                }
                if (!ok) {  // half of this PV was issued: track it so the drain below covers it
                    mma_commit(bar(B_OFULL));
                    last_bar = B_OFULL; last_par = it & 1;
                    break;
                }
                mma_commit(bar(B_OFULL));
                mma_commit(bar(B_VEMPTY));
                last_bar = B_VEMPTY; last_par = it & 1;
            }
            if (sh->abort && last_bar >= 0) drain_wait(bar(last_bar), last_par, p);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int r = threadIdx.x;  // row within the tile == tensor-memory lane
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t t_s = t_lane + C::TMEM_S, t_o = t_lane + C::TMEM_O;
        // global position of this thread's query row
        long i;
        bool row_valid;
        if (grows) {
            const int gr = q_tile * BM + r;
            row_valid = gr < p.n_global;
            i = row_valid ? p.globals[gr] : 0;
        } else {
            i = (long)q_tile * BM + r;
            row_valid = i < p.S;
        }
        // allowed key interval of this row for the window part of the mask
        long lo = 0, hi = p.S - 1;
        if (!grows) {
            if (p.kind == ATTN_MASK_CAUSAL) hi = i;
            else if (p.kind == ATTN_MASK_CAUSAL_SLIDING) { lo = i - p.window; hi = i; }
            else if (p.kind == ATTN_MASK_SLIDING || p.kind == ATTN_MASK_LOCAL_GLOBAL) { lo = i - p.window; hi = i + p.window; }
            if (hi > p.S - 1) hi = p.S - 1;
        }
        const bool lg = LG && !grows;
        const float sl2 = p.scale_log2;
        const float mL = (BIAS != BIAS_NONE) ? p.alibi[a] * 1.4426950408889634f : 0.f;  // ALiBi slope, log2 units
        const bool causal_kind = p.kind == ATTN_MASK_CAUSAL || p.kind == ATTN_MASK_CAUSAL_SLIDING;
        // bias matrix: this row's plane ([Bb, Hb] broadcast over batch / query heads)
        const size_t bplane = (BIAS == BIAS_MATRIX)
                                  ? (size_t)(p.bias_Bb == 1 ? 0 : b) * p.bias_Hb + (p.bias_Hb == 1 ? 0 : a)
                                  : 0;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int it = 0; it < n_iter; ++it) {
            uint4 bv[BIAS == BIAS_MATRIX ? 16 : 1];  // this row's bias for the tile (issued before the S wait)
            if constexpr (BIAS == BIAS_MATRIX) {
                if (!is_gathered(it)) {  // a gathered tile reads its scattered keys' bias in pass 1
                    const long c0 = (long)band_tile(band_index(it)) * BN;
                    const uint16_t* brow = (row_valid && i < p.S)
                                               ? p.bias + (bplane * (size_t)p.S + (size_t)i) * (size_t)p.bias_ld + c0
                                               : nullptr;
                    load_bias_row(bv, brow, (int)min((long)BN, (long)p.S - c0));
                }
            }
            // ---- mask of this tile (decided once per tile; FULL tiles evaluate no predicate).  It does
            // not depend on S, so it is worked out before the wait for S (the global-key bits of a
            // local + global tile are loaded here and merged in after the wait).
            bool partial = true;
            const bool gathered = is_gathered(it);
            int gcols = BN;      // gathered tiles: columns holding keys (all allowed: they lie outside the band)
            TileMask mk{0, -1, 0u, 0u, 0u, 0u};
            uint4 g4 = make_uint4(0u, 0u, 0u, 0u);
            if (!gathered) {
                const int t = band_tile(band_index(it));
                const long c0 = (long)t * BN;
                if constexpr (BN == KT) {
                    partial = t < full_begin || t >= full_end;
                } else {
                    // 64-key tiles: FULL when every row of the warp (rows past the sequence or the
                    // global list are never stored) sees the whole tile through its window interval;
                    // decided per warp, as the mask forms are
                    partial = !__all_sync(0xffffffffu, !row_valid || (lo <= c0 && hi >= c0 + BN - 1));
                }
                if (partial) {
                    mk.a0 = (int)max(-1L, min((long)BN, lo - c0));
                    mk.a1 = (int)max(-1L, min((long)BN, hi - c0));
                    if (lg) {
                        if constexpr (BN == KT) {
                            g4 = __ldg(reinterpret_cast<const uint4*>(p.global_bits + 4 * t));
                        } else {  // the tile's 64 positions are words 2t, 2t + 1 of the per-tile bits
                            const uint2 g2 = __ldg(reinterpret_cast<const uint2*>(p.global_bits + 2 * t));
                            g4 = make_uint4(g2.x, g2.y, 0u, 0u);
                        }
                    }
                }
            } else {
                gcols = gathered_cols(gat_index(it));
                mk.a1 = gcols - 1;
            }
            // no lower bound inside the tile (causal diagonal tiles, the upper edge of a window): the
            // cheap mask form, when every row of the warp qualifies (for local + global only on tiles
            // holding no global key, whose columns past the window would be allowed)
            const bool no_gkeys = !lg || (g4.x | g4.y | g4.z | g4.w) == 0u;
            const bool upper = no_gkeys && !gathered && __all_sync(0xffffffffu, partial && mk.a0 <= 0);
            // the general form (and every partial tile of the biased passes, which take no other form):
            // the interval and the global keys as column bits
            const bool bits = partial && !gathered && (!upper || BIAS != BIAS_NONE);
            if (bits) {
                mk.w0 = interval_word(mk.a0, mk.a1, 0);
                mk.w1 = interval_word(mk.a0, mk.a1, 1);
                if constexpr (BN == KT) {
                    mk.w2 = interval_word(mk.a0, mk.a1, 2);
                    mk.w3 = interval_word(mk.a0, mk.a1, 3);
                }
            }
            // warp-uniform exit: the tensor-memory accesses below are warp-collective
            if (!__all_sync(0xffffffffu, wait_bounded(bar(B_SFULL), it & 1, sh, p, ERR_SOFTMAX))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // global-row items: a warp none of whose rows is a global row (padding of the gathered
            // query tile) has nothing to compute; it still takes part in every phase of the P
            // barriers.  Its P rows keep stale values, which reach only O rows that are never stored
            // (the rows of P V are independent of one another).
            if (LG && grows && !__any_sync(0xffffffffu, row_valid)) {
                mbar_arrive(bar(B_PFULL));
                mbar_arrive(bar(B_PFULL1));
                continue;
            }
            if (lg && bits) {
                mk.w0 |= g4.x; mk.w1 |= g4.y; mk.w2 |= g4.z; mk.w3 |= g4.w;
            }
            // ---- pass 1: row max of the (masked) scores, in log2 units
            float mx;
            float base = 0.f;  // ALiBi: i - (first key of this tile); band tiles only (no local + global)
            // gathered tile under ALiBi: the key position of column c (the padding columns are masked)
            auto gpos_f = [&](int c) -> float { return c < gcols ? (float)outside_key(gat_index(it) * BN + c) : 0.f; };
            if constexpr (ALIBI) {
                base = (float)(i - (long)band_tile(band_index(it)) * BN);
                if (LG && gathered)
                    mx = narrow_row_max_alibi(t_s, (gcols + 31) >> 5, mk.a1, sl2, mL, (float)i, gpos_f);
                else if (causal_kind)
                    mx = partial ? tile_row_max_alibi<MASK_ANY, false>(t_s, mk, sl2, mL, base)
                                 : tile_row_max_alibi<MASK_NONE, false>(t_s, mk, sl2, mL, base);
                else
                    mx = partial ? tile_row_max_alibi<MASK_ANY, true>(t_s, mk, sl2, mL, base)
                                 : tile_row_max_alibi<MASK_NONE, true>(t_s, mk, sl2, mL, base);
            } else if constexpr (BIAS == BIAS_MATRIX) {
                if (LG && gathered) {
                    const uint16_t* brow0 =
                        (row_valid && i < p.S) ? p.bias + (bplane * (size_t)p.S + (size_t)i) * (size_t)p.bias_ld : nullptr;
                    mx = narrow_row_max_matbias(t_s, (gcols + 31) >> 5, mk.a1, sl2, brow0,
                                                [&](int c) -> long { return outside_key(gat_index(it) * BN + c); });
                } else {
                    mx = partial ? tile_row_max_matbias<MASK_ANY>(t_s, mk, sl2, bv)
                                 : tile_row_max_matbias<MASK_NONE>(t_s, mk, sl2, bv);
                }
            } else {
                if constexpr (LG) {
                    if (gathered) mx = narrow_row_max(t_s, (gcols + 31) >> 5, mk.a1);
                    else
                        mx = !partial ? tile_row_max<MASK_NONE, BN>(t_s, mk)
                             : upper ? tile_row_max<MASK_UPPER, BN>(t_s, mk) : tile_row_max<MASK_ANY, BN>(t_s, mk);
                } else {
                    mx = !partial ? tile_row_max<MASK_NONE, BN>(t_s, mk)
                         : upper ? tile_row_max<MASK_UPPER, BN>(t_s, mk) : tile_row_max<MASK_ANY, BN>(t_s, mk);
                }
                mx *= sl2;  // scale > 0 keeps the order; -inf stays -inf
                if constexpr (BIAS == BIAS_ALIBI_MMA) {
                    // the tile's constant part of the bias, m_a (c0 - i), in log2 units
                    base = mL * (float)((long)band_tile(band_index(it)) * BN - i);
                    mx += base;  // -inf stays -inf
                }
            }
            // ---- running max, with the lazy rescale
            const bool grow = mx > m + RESCALE_THRESHOLD;  // false when mx is -inf; true on the first finite max
            const float m_new = grow ? mx : m;
            const float ref = (m_new == -INFINITY) ? 0.f : m_new;
            // O *= alpha (rows whose max grew; rare) and l *= alpha.  O is complete up to PV(it-1): the
            // wait for S(it) covers it, because the MMA thread issues QK(it) after PV(it-1).
            auto fix = [&]() {
                float alpha = 1.f;
                if (grow) alpha = ex2(m - m_new);  // exp2(-inf) = 0 on the first finite max
                const bool fix_o = grow && it > 0 && m != -INFINITY;
                if (__any_sync(0xffffffffu, fix_o)) {
                    const float f = fix_o ? alpha : 1.f;
#pragma unroll 1
                    for (int c = 0; c < D / 16; ++c) {  // 16 columns at a time: few registers live
                        uint32_t o[16];
                        tmem_ld16(t_o + c * 16, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st16(t_o + c * 16, o);
                    }
                }
                l *= alpha;
                m = m_new;
            };
            auto no_fix = []() {};
            // ---- pass 2: P = exp2(s * scale * log2 e - m), row sum, bf16 P over the S columns
            float sum;
            if constexpr (ALIBI && F8) {  // E4M3 P
                fix();
                if (LG && gathered)
                    sum = narrow_exp_store_alibi_e4m3(t_s, (gcols + 31) >> 5, mk.a1, sl2, ref, mL, (float)i, gpos_f,
                                                      bar(B_PFULL));
                else if (causal_kind)
                    sum = partial ? tile_exp_store_alibi_e4m3<MASK_ANY, false>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL))
                                  : tile_exp_store_alibi_e4m3<MASK_NONE, false>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL));
                else
                    sum = partial ? tile_exp_store_alibi_e4m3<MASK_ANY, true>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL))
                                  : tile_exp_store_alibi_e4m3<MASK_NONE, true>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL));
            } else if constexpr (ALIBI) {
                fix();
                if (LG && gathered)
                    sum = narrow_exp_store_alibi(t_s, (gcols + 31) >> 5, mk.a1, sl2, ref, mL, (float)i, gpos_f, bar(B_PFULL));
                else if (causal_kind)
                    sum = partial ? tile_exp_store_alibi<MASK_ANY, false>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL))
                                  : tile_exp_store_alibi<MASK_NONE, false>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL));
                else
                    sum = partial ? tile_exp_store_alibi<MASK_ANY, true>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL))
                                  : tile_exp_store_alibi<MASK_NONE, true>(t_s, mk, sl2, ref, mL, base, bar(B_PFULL));
            } else if constexpr (BIAS == BIAS_MATRIX) {
                fix();
                // x is already scaled, biased and masked
                if (LG && gathered)
                    sum = F8 ? narrow_exp_store_e4m3(t_s, (gcols + 31) >> 5, mk.a1, 1.f, ref, bar(B_PFULL), no_fix)
                             : narrow_exp_store(t_s, (gcols + 31) >> 5, mk.a1, 1.f, ref, bar(B_PFULL), no_fix);
                else if constexpr (F8)
                    sum = tile_exp_store_e4m3<MASK_NONE>(t_s, mk, 1.f, ref, bar(B_PFULL));
                else
                    sum = tile_exp_store<MASK_NONE>(t_s, mk, 1.f, ref, bar(B_PFULL), no_fix);
            } else if constexpr (F8) {
                if (LG && gathered) {
                    sum = narrow_exp_store_e4m3(t_s, (gcols + 31) >> 5, mk.a1, sl2, ref, bar(B_PFULL), fix);
                } else {
                    fix();
                    sum = !partial ? tile_exp_store_e4m3<MASK_NONE>(t_s, mk, sl2, ref, bar(B_PFULL))
                          : upper ? tile_exp_store_e4m3<MASK_UPPER>(t_s, mk, sl2, ref, bar(B_PFULL))
                                  : tile_exp_store_e4m3<MASK_ANY>(t_s, mk, sl2, ref, bar(B_PFULL));
                }
            } else {
                const float r_eff = (BIAS == BIAS_ALIBI_MMA) ? ref - base : ref;  // x = s sl2 + base - ref
                if (LG && gathered)
                    sum = narrow_exp_store(t_s, (gcols + 31) >> 5, mk.a1, sl2, r_eff, bar(B_PFULL), fix);
                else if constexpr (BN == 64)
                    sum = !partial ? tile_exp_store_n64<MASK_NONE>(t_s, mk, sl2, r_eff, bar(B_PFULL), fix)
                          : upper ? tile_exp_store_n64<MASK_UPPER>(t_s, mk, sl2, r_eff, bar(B_PFULL), fix)
                                  : tile_exp_store_n64<MASK_ANY>(t_s, mk, sl2, r_eff, bar(B_PFULL), fix);
                else
                    sum = !partial ? tile_exp_store<MASK_NONE>(t_s, mk, sl2, r_eff, bar(B_PFULL), fix)
                          : upper ? tile_exp_store<MASK_UPPER>(t_s, mk, sl2, r_eff, bar(B_PFULL), fix)
                                  : tile_exp_store<MASK_ANY>(t_s, mk, sl2, r_eff, bar(B_PFULL), fix);
            }
            l += sum;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL1));
        }
        // ---- epilogue
        if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(B_OFULL), (n_iter - 1) & 1, sh, p, ERR_SOFTMAX));
        tc_fence_after();
        ok = named_bar_and(1, 128, ok);  // the same decision in all four softmax warps
        if (ok) {
            // o_scale: the V descale of E4M3 inputs (bf16 inputs have none; callers may leave it 0)
            const float inv_l = l > 0.f ? (F8 ? p.o_scale : 1.f) / l : 0.f;
            const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            // band items of local + global whose tile holds global rows leave those rows to the
            // global-row items and store the others directly
            const bool tile_has_g = LG && !grows && (flags & ATTN_WORK_HAS_GLOBAL_ROWS);
            const bool skip_g = tile_has_g && ((__ldg(p.global_bits + 4 * q_tile + (r >> 5)) >> (r & 31)) & 1u);
            if (tile_has_g) {
                store_row_direct<D>(t_o, static_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.S + i) * D, inv_l,
                                    row_valid && !skip_g);
            } else if (!grows) {
                // O row -> bf16 -> 128B-swizzled staging in the (now idle) Q buffer -> TMA store
                uint8_t* stage = smem + C::OFF_Q;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c * 32, o);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
                    const int sub = c >> 1;              // 64-column block
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int chunk = (c & 1) * 4 + q;  // 16-byte chunk within the 128-byte row
                        uint4* dst = reinterpret_cast<uint4*>(stage + sub * C::OSUB + r * 128 + ((chunk ^ (r & 7)) << 4));
                        *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(1, 128);
                if (threadIdx.x == 0) {
                    // O is bf16 (64 columns per 128-byte block); with E4M3 inputs the staging runs on
                    // into the (idle) K buffer that follows the Q buffer
                    for (int s = 0; s < D / 64; ++s) tma_store_3d(&p.tm_o, s_q + s * C::OSUB, s * 64, q_tile * BM, bh);
                    tma_store_commit_and_wait_read();
                }
            } else if (p.n_chunks == 1) {
                // global rows: scattered row stores; rows past the list skip them
                store_row_direct<D>(t_o, static_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.S + i) * D, inv_l, row_valid);
            } else {
                // one key chunk of a global row: fp32 partial O (normalised by this chunk's
                // sum) and partial LSE, merged below by the chunk that finishes last
                const size_t slot = ((size_t)bh * p.n_global + (q_tile * BM + r)) * p.n_chunks + n_gt;
                float4* dst = reinterpret_cast<float4*>(p.part_o + slot * D);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_o + c * 32, o);
                    tmem_wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[c * 8 + q] = make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                                         __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
                    }
                }
                if (row_valid) p.part_lse[slot] = lse;
            }
            if (p.lse && row_valid && !skip_g && !(grows && p.n_chunks > 1)) p.lse[(size_t)bh * p.S + i] = lse;
        }
        if (grows && p.n_chunks > 1) {
            // Count this chunk in (also after an abort, so that the counter returns to 0); the chunk
            // that finishes last merges every chunk of the row tile and resets the counter.
            __threadfence();  // this thread's partial stores, before the arrival
            named_bar_sync(1, 128);
            unsigned* counter = p.counters + (size_t)bh * p.n_gtiles + q_tile;
            if (threadIdx.x == 0) sh->merge_last = atomicAdd(counter, 1u) == (unsigned)(p.n_chunks - 1);
            named_bar_sync(1, 128);
            if (sh->merge_last) {
                __threadfence();
                // one warp per global row of the tile (the four softmax warps take turns)
                const int n_rows = min(BM, p.n_global - q_tile * BM);
                for (int rr = warp; rr < n_rows; rr += 4) {
                    const long ig = __ldg(p.globals + q_tile * BM + rr);
                    merge_global_row<D>(p, ((size_t)bh * p.n_global + (q_tile * BM + rr)) * p.n_chunks,
                                        static_cast<__nv_bfloat16*>(p.o) + ((size_t)bh * p.S + ig) * D,
                                        p.lse ? p.lse + (size_t)bh * p.S + ig : nullptr, lane);
                }
                if (threadIdx.x == 0) *counter = 0u;
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

template <int D, int BIAS, bool F8 = false, bool LG = false, int BN = 128>
cudaError_t launch(const TcParams& p, int n_items, cudaStream_t stream) {
    using C = Cfg<D, BIAS, F8, BN>;
    cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(attn_fwd_tc_kernel<D, BIAS, F8, LG, BN>), C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attn_fwd_tc_kernel<D, BIAS, F8, LG, BN><<<n_items, NTHREADS, C::SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_forward(const TcParams& p, int d, int n_items, cudaStream_t stream) {
    if (n_items <= 0) return cudaSuccess;
    const bool causal = p.kind == ATTN_MASK_CAUSAL || p.kind == ATTN_MASK_CAUSAL_SLIDING;
    if (p.fp8) {  // E4M3 inputs: d = 128 or 64 (checked by the host)
        const bool lg = p.kind == ATTN_MASK_LOCAL_GLOBAL && p.n_global > 0;
        if (d == 128 && p.alibi)  // ALiBi added per element for every kind (no bf16 bias product with E4M3 operands)
            return lg ? launch<128, BIAS_ALIBI_ELEM, true, true>(p, n_items, stream)
                      : launch<128, BIAS_ALIBI_ELEM, true>(p, n_items, stream);
        if (d == 128) {
            if (p.bias) return lg ? launch<128, BIAS_MATRIX, true, true>(p, n_items, stream)
                                  : launch<128, BIAS_MATRIX, true>(p, n_items, stream);
            return lg ? launch<128, BIAS_NONE, true, true>(p, n_items, stream)
                      : launch<128, BIAS_NONE, true>(p, n_items, stream);
        }
        if (d == 64) {  // 64-byte rows: the 64-byte swizzle layout
            if (p.alibi) return lg ? launch<64, BIAS_ALIBI_ELEM, true, true>(p, n_items, stream)
                                   : launch<64, BIAS_ALIBI_ELEM, true>(p, n_items, stream);
            if (p.bias) return lg ? launch<64, BIAS_MATRIX, true, true>(p, n_items, stream)
                                  : launch<64, BIAS_MATRIX, true>(p, n_items, stream);
            return lg ? launch<64, BIAS_NONE, true, true>(p, n_items, stream)
                      : launch<64, BIAS_NONE, true>(p, n_items, stream);
        }
        return cudaErrorInvalidValue;
    }
    if (p.bias) {  // a bias matrix (bf16 inputs; checked by the host)
        if (p.kind == ATTN_MASK_LOCAL_GLOBAL && p.n_global > 0) {
            if (d == 128) return launch<128, BIAS_MATRIX, false, true>(p, n_items, stream);
            if (d == 64) return launch<64, BIAS_MATRIX, false, true>(p, n_items, stream);
            return cudaErrorInvalidValue;
        }
        if (d == 128) return launch<128, BIAS_MATRIX>(p, n_items, stream);
        if (d == 64) return launch<64, BIAS_MATRIX>(p, n_items, stream);
        return cudaErrorInvalidValue;
    }
    if (p.kind == ATTN_MASK_LOCAL_GLOBAL && p.n_global > 0 && p.alibi) {  // gathered keys under ALiBi
        if (d == 128) return launch<128, BIAS_ALIBI_ELEM, false, true>(p, n_items, stream);
        if (d == 64) return launch<64, BIAS_ALIBI_ELEM, false, true>(p, n_items, stream);
        return cudaErrorInvalidValue;
    }
    if (p.alibi && causal) {
        if (d == 128) return launch<128, BIAS_ALIBI_MMA>(p, n_items, stream);
        if (d == 64) return launch<64, BIAS_ALIBI_MMA>(p, n_items, stream);
    } else if (p.alibi) {
        if (d == 128) return launch<128, BIAS_ALIBI_ELEM>(p, n_items, stream);
        if (d == 64) return launch<64, BIAS_ALIBI_ELEM>(p, n_items, stream);
    } else if (p.kind == ATTN_MASK_LOCAL_GLOBAL && p.n_global > 0) {  // gathered keys, global-row chunks
        if (d == 128) return launch<128, BIAS_NONE, false, true>(p, n_items, stream);
        if (d == 64) return launch<64, BIAS_NONE, false, true, 64>(p, n_items, stream);
    } else {
        if (d == 128) return launch<128, BIAS_NONE>(p, n_items, stream);
        if (d == 64) return launch<64, BIAS_NONE, false, false, 64>(p, n_items, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace attn
