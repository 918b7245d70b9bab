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
// The work is bound by HBM: every key and value byte is used by group * S_q
// query rows only.  So one CTA takes ALL query rows of one kv head's group
// (a GQA/MQA group reads its shared cache once, "第 8 章", 8.2.2 on MQA's
// single HBM read for h heads) and the tensor-core products are transposed so
// that the 128 keys of a tile fill the MMA's M dimension and the packed query
// rows its N dimension (NP = 16, 32 or 64 columns):
//
//   S^T [128 keys x NP]  = K_tile [128 x d]  . Q^T [d x NP]      (both K-major)
//   O^T [d x NP]        += V_tile^T [d x 128] . P^T [128 x NP]   (V MN-major)
//
//   warp 4 (producer) : TMA loads of the packed Q rows (once) and of the K and
//                       V tiles into a STAGES-deep ring of 128B-swizzled tiles.
//   warp 5 (MMA)      : one thread issues QK(n+1) before PV(n) so that the
//                       softmax of tile n+1 overlaps the PV of tile n (S^T is
//                       double-buffered in tensor memory, P^T in shared memory).
//   warps 0-3         : thread t owns key t of the tile (tensor-memory lane t)
//                       and, for O^T, component t of d.  Row maxima over the
//                       128 keys come from warp reductions plus a 4-warp
//                       exchange; the running max/sum use exp2 on log2(e)-
//                       prescaled scores with the lazy rescale (only when a
//                       row's max grew by more than 2^8).  P^T goes to shared
//                       memory in the MMA's K-major swizzled layout.
//
// Long caches are split into chunks of key tiles (several CTAs per sequence
// and kv head); each chunk writes its O normalised by its own sum and its
// LSE, and the last CTA of the sequence to finish (an atomic arrival counter
// that wraps back to zero) combines them with weights e^{LSE_c - LSE}.
//
// Stale cache entries (positions >= cache_len[b]) are never used: their scores
// are masked, and the V rows of the last tile past the cache length are zeroed
// in shared memory before the PV product (0 * NaN would otherwise be NaN).
// Every mbarrier wait is bounded by the watchdog limit (see attn_fwd_tc.cu).
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "schedule.h"
#include "sm103_ptx.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int BN = 128;         // keys per tile (the MMA's M)
constexpr int NTHREADS = 192;   // 4 softmax warps + producer + MMA
constexpr int WARP_PRODUCER = 4;
constexpr int WARP_MMA = 5;
constexpr int MAX_STAGES = 4;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
constexpr int SMEM_LIMIT = 227 * 1024;

enum : int { ERR_PRODUCER = 1, ERR_MMA = 2, ERR_SOFTMAX = 4 };

template <int D, int NP>
struct DCfg {
    static constexpr int TB = BN * D * 2;         // one K or V tile
    static constexpr int SUB = BN * 128;          // one 64-column block of a K/V tile
    static constexpr int QB = NP * 128;           // one 64-column block of the Q rows
    static constexpr int PB = NP * 128;           // one 64-key half of a P^T buffer
    static constexpr int ZERO = (D == 64) ? SUB : 0;  // rows 64..127 of V^T when d = 64 (zeros)
    static constexpr int CTL = 8192;
    static constexpr int FIXED = NP * D * 2 + 2 * 2 * PB + ZERO + CTL + 1024;
    static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED) / (2 * TB);
    static constexpr int STAGES = STAGES_FIT > MAX_STAGES ? MAX_STAGES : STAGES_FIT;
    static_assert(STAGES >= 2, "shared memory");
    static constexpr int OFF_V = 0;
    static constexpr int OFF_K = OFF_V + STAGES * TB;
    static constexpr int OFF_Z = OFF_K + STAGES * TB;
    static constexpr int OFF_Q = OFF_Z + ZERO;
    static constexpr int OFF_P = OFF_Q + NP * D * 2;
    static constexpr int OFF_CTL = OFF_P + 2 * 2 * PB;
    static constexpr int SMEM_ALLOC = OFF_CTL + CTL + 1024;
    static constexpr uint32_t TMEM_COLS = (3 * NP <= 64) ? 64 : (3 * NP <= 128) ? 128 : 256;
    static constexpr uint32_t TMEM_S = 0;       // S^T buffers: columns [0, NP) and [NP, 2 NP)
    static constexpr uint32_t TMEM_O = 2 * NP;  // O^T: columns [2 NP, 3 NP)
    // merge weights of a split sequence live in the (idle) K ring at the end
    static constexpr int MAX_MERGE_CHUNKS = STAGES * TB / (NP * 4);
    static_assert(MAX_MERGE_CHUNKS >= kDecodeMaxChunksPerSeq, "merge weights must fit the K ring");
};

enum Bar {
    B_Q = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + MAX_STAGES,
    B_VFULL = B_KEMPTY + MAX_STAGES,
    B_VEMPTY = B_VFULL + MAX_STAGES,
    B_SFULL = B_VEMPTY + MAX_STAGES,  // 2: S^T buffer ready (MMA commit)
    B_PFULL = B_SFULL + 2,            // 2: P^T buffer written, S^T buffer read (128 arrivals)
    B_PFREE = B_PFULL + 2,            // 2: PV done with the P^T buffer (MMA commit)
    B_OFULL = B_PFREE + 2,            // every PV (MMA commit)
    NBAR = B_OFULL + 1
};

template <int NP>
struct DShared {
    uint64_t bar[NBAR];
    uint32_t tmem_base;
    volatile int abort;
    int is_last;
    int flag[2];          // a row of this tile needs O and l rescaled
    int wmax[2][4][NP];   // per-warp tile maxima, order-preserving int encoding
    int lo[NP], hi[NP];   // allowed key interval of each packed row
    float m[NP], alpha[NP];
    float lsum[4][NP];
    float l[NP], lse[NP];
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

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <int D, int NP>
__global__ void __launch_bounds__(NTHREADS, 1) attn_decode_kernel(const __grid_constant__ DecodeParams p) {
    using C = DCfg<D, NP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    DShared<NP>* sh = reinterpret_cast<DShared<NP>*>(smem + C::OFF_CTL);
    const uint32_t s_v = smem_u32(smem + C::OFF_V);
    const uint32_t s_k = smem_u32(smem + C::OFF_K);
    const uint32_t s_z = smem_u32(smem + C::OFF_Z);
    const uint32_t s_q = smem_u32(smem + C::OFF_Q);
    const uint32_t s_p = smem_u32(smem + C::OFF_P);
    auto bar = [&](int b) { return smem_u32(&sh->bar[b]); };
    const Watch wd{&sh->abort, p.err, p.watchdog_ns};

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work of this CTA: sequence b, kv head g, key tiles [t0, t0 + n_iter)
    const int x = blockIdx.x, g = blockIdx.y;
    int b = 0;
    {
        int lo = 0, hi = p.B - 1;  // last sequence whose first chunk is <= x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.chunk_prefix[mid] <= x) lo = mid; else hi = mid - 1;
        }
        b = lo;
    }
    const int chunk = x - p.chunk_prefix[b];
    const int n_chunks = p.chunk_prefix[b + 1] - p.chunk_prefix[b];
    const int L = p.len[b];
    const bool sliding = p.kind == ATTN_MASK_CAUSAL_SLIDING;
    const int t_lo = sliding ? max(0, L - p.S_q - p.window) / BN : 0;
    const int t_hi = (L + BN - 1) / BN;
    const int t0 = t_lo + chunk * p.tiles_per_chunk;
    const int n_iter = min(t_hi, t0 + p.tiles_per_chunk) - t0;  // >= 1 by construction of the chunks
    const int bkv = b * p.Hkv + g;
    const int row0 = (b * p.Hq + g * p.group) * p.S_q;  // first packed query row
    // tightest bounds over the valid rows: a tile inside [max_lo, min_hi] needs no mask
    const int max_lo = sliding ? L - 1 - p.window : 0;
    const int min_hi = p.kind == ATTN_MASK_FULL ? L - 1 : L - p.S_q;
    const int tail = (L % BN == 0) ? 0 : L % BN;  // valid keys of the last cache tile (0 = whole)

    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i == B_PFULL || i == B_PFULL + 1) ? 128u : 1u);
        sh->abort = 0;
        sh->flag[0] = sh->flag[1] = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < NP) {
        const int r = threadIdx.x;
        int lo = 0, hi = L - 1;
        if (r < p.rows && p.kind != ATTN_MASK_FULL) {
            const int pos = L - p.S_q + r % p.S_q;  // position of this query row
            hi = pos;
            if (sliding) lo = max(0, pos - p.window);
        }
        sh->lo[r] = lo;
        sh->hi[r] = hi;
        sh->m[r] = -INFINITY;
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

    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q), NP * D * 2);
            for (int s = 0; s < D / 64; ++s) tma_load_2d(s_q + s * C::QB, &p.tm_q, bar(B_Q), s * 64, row0);
            int k_loaded = 0, v_loaded = 0;
            bool ok = true;
            for (int n = 0; n < n_iter && ok; ++n) {
                const int st = n % C::STAGES, round = n / C::STAGES;
                const int key = (t0 + n) * BN;
                if (n >= C::STAGES && !(ok = wait_bounded(bar(B_KEMPTY + st), (round - 1) & 1, wd, ERR_PRODUCER)))
                    break;
                mbar_arrive_expect_tx(bar(B_KFULL + st), C::TB);
                for (int s = 0; s < D / 64; ++s)
                    tma_load_3d(s_k + st * C::TB + s * C::SUB, &p.tm_k, bar(B_KFULL + st), s * 64, key, bkv);
                k_loaded = n + 1;
                if (n >= C::STAGES && !(ok = wait_bounded(bar(B_VEMPTY + st), (round - 1) & 1, wd, ERR_PRODUCER)))
                    break;
                mbar_arrive_expect_tx(bar(B_VFULL + st), C::TB);
                for (int s = 0; s < D / 64; ++s)
                    tma_load_3d(s_v + st * C::TB + s * C::SUB, &p.tm_v, bar(B_VFULL + st), s * 64, key, bkv);
                v_loaded = n + 1;
            }
            if (sh->abort) {  // let the copies in flight land before the CTA exits
                drain_wait(bar(B_Q), 0, wd);
                for (int n = max(0, k_loaded - C::STAGES); n < k_loaded; ++n)
                    drain_wait(bar(B_KFULL + n % C::STAGES), (n / C::STAGES) & 1, wd);
                for (int n = max(0, v_loaded - C::STAGES); n < v_loaded; ++n)
                    drain_wait(bar(B_VFULL + n % C::STAGES), (n / C::STAGES) & 1, wd);
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer (lane 0) + V tail zeroing (warp)
        constexpr uint32_t idesc_qk = idesc_bf16_f32_ab(BN, NP, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32_ab(BN, NP, true, false);
        // V^T as an MN-major A operand: d is contiguous; the second 64-row block of d
        // (or the zero block when d = 64) sits LBO bytes after the first
        auto v_lbo = [&](int st) -> uint32_t {
            return D == 128 ? (uint32_t)C::SUB : (uint32_t)(s_z - (s_v + st * C::TB));
        };
        int last_bar = -1, last_par = 0;  // the last commit (drained after an abort)
        auto issue_qk = [&](int n) {
            const int st = n % C::STAGES;
            const uint32_t t_s = tmem + C::TMEM_S + (n & 1) * NP;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t a = s_k + st * C::TB + (k >> 2) * C::SUB + (k & 3) * 32;
                const uint32_t bq = s_q + (k >> 2) * C::QB + (k & 3) * 32;
                mma_ss(t_s, sdesc_sw128(a, 16, 1024), sdesc_sw128(bq, 16, 1024), idesc_qk, k > 0);
            }
            mma_commit(bar(B_SFULL + (n & 1)));
            mma_commit(bar(B_KEMPTY + st));
            last_bar = B_SFULL + (n & 1);
            last_par = (n >> 1) & 1;
        };
        bool ok = true;
        if (lane == 0) {
            ok = wait_bounded(bar(B_Q), 0, wd, ERR_MMA) && wait_bounded(bar(B_KFULL), 0, wd, ERR_MMA);
            if (ok) {
                tc_fence_after();
                issue_qk(0);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // The whole warp runs the loop (the exit is warp-uniform); lane 0 waits and issues.
        for (int n = 0; n < n_iter && ok; ++n) {
            const int st = n % C::STAGES;
            if (lane == 0) {
                if (n + 1 < n_iter) {
                    ok = wait_bounded(bar(B_KFULL + (n + 1) % C::STAGES), ((n + 1) / C::STAGES) & 1, wd, ERR_MMA);
                    if (ok) {
                        tc_fence_after();
                        issue_qk(n + 1);  // S^T buffer (n+1)&1 was released by the softmax before PV(n-1)
                    }
                }
                if (ok) ok = wait_bounded(bar(B_PFULL + (n & 1)), (n >> 1) & 1, wd, ERR_MMA);
                if (ok) ok = wait_bounded(bar(B_VFULL + st), (n / C::STAGES) & 1, wd, ERR_MMA);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (tail != 0 && t0 + n == t_hi - 1) {
                // the last cache tile: zero the V rows at and past the cache length.  Every lane
                // observes the completed copy itself (the phase cannot advance before this PV).
                const bool seen = lane == 0 || wait_bounded(bar(B_VFULL + st), (n / C::STAGES) & 1, wd, ERR_MMA);
                if (!__all_sync(0xffffffffu, seen)) {
                    ok = false;
                    break;
                }
                uint8_t* vt = smem + C::OFF_V + st * C::TB;
                const int nbytes = (BN - tail) * 128;
                for (int s = 0; s < D / 64; ++s)
                    for (int i = lane * 16; i < nbytes; i += 32 * 16)
                        *reinterpret_cast<uint4*>(vt + s * C::SUB + tail * 128 + i) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t t_o = tmem + C::TMEM_O;
                const uint32_t pb = s_p + (n & 1) * 2 * C::PB;
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint32_t a = s_v + st * C::TB + k * 16 * 128;  // 16 keys of 128-byte rows
                    const uint32_t bp = pb + (k >> 2) * C::PB + (k & 3) * 32;
                    mma_ss(t_o, sdesc_sw128(a, v_lbo(st), 1024), sdesc_sw128(bp, 16, 1024), idesc_pv,
                           (n > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_OFULL));
                mma_commit(bar(B_VEMPTY + st));
                mma_commit(bar(B_PFREE + (n & 1)));
                last_bar = B_PFREE + (n & 1);
                last_par = (n >> 1) & 1;
            }
        }
        if (lane == 0 && sh->abort && last_bar >= 0) drain_wait(bar(last_bar), last_par, wd);
    } else {
        // ------------------------------------------------------------ softmax + epilogue (warps 0-3)
        const int t = threadIdx.x;  // key within the tile == tensor-memory lane; d index of O^T
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        // waits of the four softmax warps end with the same outcome in all of them (the
        // loop below has named barriers, so every exit must be taken by all 128 threads)
        auto sm_wait = [&](int b_, uint32_t parity) {
            return named_bar_and(1, 128, wait_bounded(bar(b_), parity, wd, ERR_SOFTMAX));
        };
        float lp[NP];  // this thread's share of every row's sum
#pragma unroll
        for (int r = 0; r < NP; ++r) lp[r] = 0.f;
        bool ok = true;
        for (int n = 0; n < n_iter; ++n) {
            const int par = n & 1;
            if (!sm_wait(B_SFULL + par, (n >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int j = (t0 + n) * BN + t;  // this thread's key
            const bool full = (t0 + n) * BN >= max_lo && (t0 + n) * BN + BN - 1 <= min_hi;
            const uint32_t t_s = t_lane + C::TMEM_S + par * NP;
            // ---- pass 1: masked tile maxima of every row
#pragma unroll
            for (int c = 0; c < NP / 16; ++c) {
                uint32_t v[16];
                tmem_ld16(t_s + c * 16, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r = c * 16 + e;
                    float s = __uint_as_float(v[e]);
                    if (!full && !(j >= sh->lo[r] && j <= sh->hi[r])) s = -INFINITY;
                    const int mx = __reduce_max_sync(0xffffffffu, ordered(s));
                    if (lane == 0) sh->wmax[par][warp][r] = mx;
                }
            }
            named_bar_sync(1, 128);
            if (t == 0) sh->flag[par ^ 1] = 0;  // the next tile's flag: its last readers are past this barrier
            if (t < NP) {
                const int k4 = max(max(sh->wmax[par][0][t], sh->wmax[par][1][t]),
                                   max(sh->wmax[par][2][t], sh->wmax[par][3][t]));
                const float tmax = unordered(k4) * sl2;  // -inf stays -inf (scale > 0)
                const float m_old = sh->m[t];
                const bool grow = tmax > m_old + RESCALE_THRESHOLD;  // true on the first finite max
                const float m_new = grow ? tmax : m_old;
                sh->m[t] = m_new;
                sh->alpha[t] = grow ? ex2(m_old - m_new) : 1.f;
                if (grow && m_old != -INFINITY) sh->flag[par] = 1;
            }
            named_bar_sync(1, 128);
            if (sh->flag[par]) {
                // some row's max grew: scale the sums and (after PV(n-1)) the O^T columns
#pragma unroll
                for (int r = 0; r < NP; ++r) lp[r] *= sh->alpha[r];
                if (!sm_wait(B_OFULL, (n - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < NP / 16; ++c) {
                    uint32_t o[16];
                    tmem_ld16(t_lane + C::TMEM_O + c * 16, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * sh->alpha[c * 16 + e]);
                    tmem_st16(t_lane + C::TMEM_O + c * 16, o);
                }
                tmem_wait_st();
            }
            // ---- the P^T buffer of this parity is free once PV(n-2) is done
            if (n >= 2 && !sm_wait(B_PFREE + par, ((n >> 1) - 1) & 1)) {
                ok = false;
                break;
            }
            // ---- pass 2: P = exp2(s * scale * log2 e - m) -> bf16 P^T (K-major, 128B swizzle)
            const uint32_t pb = s_p + par * 2 * C::PB + (t >> 6) * C::PB;
            const int kk = t & 63;
#pragma unroll
            for (int c = 0; c < NP / 16; ++c) {
                uint32_t v[16];
                tmem_ld16(t_s + c * 16, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    float pr[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int r = c * 16 + e + u;
                        const bool in = full || (j >= sh->lo[r] && j <= sh->hi[r]);
                        const float m = sh->m[r];
                        pr[u] = in ? ex2(fmaf(__uint_as_float(v[e + u]), sl2, -m)) : 0.f;
                        lp[r] += pr[u];
                    }
                    const uint32_t pk = pack_bf16x2(pr[0], pr[1]);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int r = c * 16 + e + u;
                        const uint32_t addr = pb + r * 128 + ((((kk >> 3) ^ (r & 7))) << 4) + (kk & 7) * 2;
                        st_shared_u16(addr, (uint16_t)(u ? (pk >> 16) : (pk & 0xffffu)));
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL + par));
        }
        // ---- epilogue
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o);
        if (ok) ok = sm_wait(B_OFULL, (n_iter - 1) & 1);  // ok is the same in all 128 threads here
        tc_fence_after();
        if (ok) {
            // every row's sum: warp sums, then the four warps
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
                sh->l[t] = l > 0.f ? 1.f / l : 0.f;
                sh->lse[t] = l > 0.f ? (sh->m[t] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
            named_bar_sync(1, 128);
            const size_t slot = (size_t)g * p.total_chunks + x;
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
                            const float val = __uint_as_float(o[e]) * sh->l[r];
                            if (n_chunks == 1) out[(size_t)(row0 + r) * D + t] = __float2bfloat16_rn(val);
                            else p.part_o[(slot * NP + r) * D + t] = val;
                        }
                    }
                }
            }
            if (t < p.rows) {
                if (n_chunks == 1) {
                    if (p.lse) p.lse[row0 + t] = sh->lse[t];
                } else {
                    p.part_lse[slot * NP + t] = sh->lse[t];
                }
            }
        }
        if (n_chunks > 1) {
            // arrival of this chunk (also after an abort, so the counter keeps wrapping to 0)
            __threadfence();
            named_bar_sync(1, 128);
            if (t == 0) sh->is_last = atomicInc(p.counters + bkv, (unsigned)(n_chunks - 1)) == (unsigned)(n_chunks - 1);
            named_bar_sync(1, 128);
            if (ok && sh->is_last) {
                __threadfence();
                // weights e^{LSE_c - LSE} of every chunk and row, in the idle K ring
                float* wts = reinterpret_cast<float*>(smem + C::OFF_K);  // [n_chunks][NP]
                const size_t slot0 = (size_t)g * p.total_chunks + p.chunk_prefix[b];
                if (t < p.rows) {
                    float M = -INFINITY;
                    for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, __ldcg(p.part_lse + (slot0 + c) * NP + t));
                    float W = 0.f;
                    for (int c = 0; c < n_chunks; ++c) {
                        const float w = __expf(__ldcg(p.part_lse + (slot0 + c) * NP + t) - M);
                        wts[c * NP + t] = w;
                        W += w;
                    }
                    const float inv = 1.f / W;
                    for (int c = 0; c < n_chunks; ++c) wts[c * NP + t] *= inv;
                    if (p.lse) p.lse[row0 + t] = M + __logf(W);
                }
                named_bar_sync(1, 128);
                if (t < D) {
                    for (int r = 0; r < p.rows; ++r) {
                        float acc = 0.f;
                        for (int c = 0; c < n_chunks; ++c)
                            acc += wts[c * NP + r] * __ldcg(p.part_o + ((slot0 + c) * NP + r) * D + t);
                        out[(size_t)(row0 + r) * D + t] = __float2bfloat16_rn(acc);
                    }
                }
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

template <int D, int NP>
cudaError_t launch(const DecodeParams& p, cudaStream_t stream) {
    using C = DCfg<D, NP>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const dim3 grid(p.total_chunks, p.Hkv);
    attn_decode_kernel<D, NP><<<grid, NTHREADS, C::SMEM_ALLOC, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int d, int np, cudaStream_t stream) {
    if (p.total_chunks <= 0) return cudaSuccess;
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
