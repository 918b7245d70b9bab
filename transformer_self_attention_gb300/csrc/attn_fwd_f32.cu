// fp32 attention forward on CUDA cores, and the self-test of the FMA-pipe exp2.
//
// The fp32 path keeps full fp32 inputs and arithmetic (TF32 tensor cores
// would round the inputs to 10 mantissa bits).  One CTA owns a tile of QT query
// rows of one (batch, head) and walks the key tiles of KT keys its rows may see,
// staged in shared memory (the next tile's loads in flight while one is
// computed); per key tile it forms the QT x KT scores (sixteen threads per row,
// KT / 16 keys each), applies the mask, updates the running max and sum of each
// row (the online softmax of "Transformer 演进与变体" (ai.icyfenix.cn), section
// Flash Attention, 在线 Softmax) and accumulates O += P V (the same sixteen
// threads per row, d / 16 columns each).  The mask is
// the plain predicate per (row, key): the window interval, and for local +
// global a global row or a global key ("Transformer 演进与变体", section 稀疏注意力);
// key tiles holding no allowed pair for any row of the tile are skipped.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn.h"
#include "kernels.h"
#include "sm103_ptx.h"

namespace attn {
namespace {

constexpr int QT = 8;            // query rows per CTA
constexpr int KT32 = 32;         // keys per tile
constexpr int TPR = 16;          // threads per query row
constexpr int F32_THREADS = QT * TPR;

// Row strides are padded so that the rows a warp works on fall in distinct banks (Q, P) and the
// keys of a row's lanes in distinct banks (K, 16-byte rows kept for the vector stores).
template <int D>
struct F32Smem {
    float q[QT][D + 1];
    float k[KT32][D + 4];
    float v[KT32][D];
    float p[QT][KT32 + 1];
};

template <int D>
__global__ void __launch_bounds__(F32_THREADS) attn_fwd_f32_kernel(F32Params p) {
    constexpr int KPT = KT32 / TPR;  // keys per thread
    constexpr int CPT = D / TPR;     // O columns per thread
    constexpr int LPT = KT32 * D / 4 / F32_THREADS;  // 16-byte K (and V) loads per thread per tile
    __shared__ __align__(16) F32Smem<D> sm;
    const int tid = threadIdx.x, r = tid / TPR, g = tid % TPR;  // row of the tile, lane within the row
    const int n_qt = (p.S + QT - 1) / QT;
    const long bh = blockIdx.x / n_qt;
    const long i0 = (long)(blockIdx.x - bh * n_qt) * QT;
    const long b = bh / p.Hq, a = bh - b * p.Hq;
    const long bkv = b * p.Hkv + a / p.group;  // g(a) = a / (Hq / Hkv)
    const float* Kh = p.k + bkv * (long)p.S * D;
    const float* Vh = p.v + bkv * (long)p.S * D;

    // this thread's query row and its allowed key interval (the window part)
    const long i = i0 + r;
    const bool row_valid = i < p.S;
    const bool lg = p.kind == ATTN_MASK_LOCAL_GLOBAL && p.n_global > 0;
    const bool g_row = lg && row_valid && p.is_global[i];
    long lo = 0, hi = p.S - 1;
    if (g_row) {
        // a global row sees every key
    } else if (p.kind == ATTN_MASK_CAUSAL) {
        hi = i;
    } else if (p.kind == ATTN_MASK_CAUSAL_SLIDING) {
        lo = i - p.window;
        hi = i;
    } else if (p.kind == ATTN_MASK_SLIDING || p.kind == ATTN_MASK_LOCAL_GLOBAL) {
        lo = i - p.window;
        hi = i + p.window;
    }
    if (hi > p.S - 1) hi = p.S - 1;
    if (!row_valid) { lo = 1; hi = 0; }  // a padding row sees nothing (never stored)
    const float slope = p.alibi ? p.alibi[a] : 0.f;

    for (int e = tid; e < QT * D; e += F32_THREADS) {
        const int rr = e / D, c = e - rr * D;
        sm.q[rr][c] = (i0 + rr < p.S) ? p.q[(bh * p.S + i0 + rr) * D + c] : 0.f;
    }
    // the tile's key range for the window part: the union of its rows' intervals
    long t_lo = 0, t_hi = p.S - 1;
    {
        const long r1 = (i0 + QT < p.S ? i0 + QT : p.S) - 1;
        if (p.kind == ATTN_MASK_CAUSAL) t_hi = r1;
        else if (p.kind == ATTN_MASK_CAUSAL_SLIDING) { t_lo = i0 - p.window; t_hi = r1; }
        else if (p.kind == ATTN_MASK_SLIDING || p.kind == ATTN_MASK_LOCAL_GLOBAL) { t_lo = i0 - p.window; t_hi = r1 + p.window; }
        if (t_lo < 0) t_lo = 0;
        if (t_hi > p.S - 1) t_hi = p.S - 1;
    }
    const bool any_g_row = __syncthreads_or(g_row && g == 0);  // also orders the Q stores
    const int n_kt = (p.S + KT32 - 1) / KT32;
    // the key tiles to visit, in order: those meeting the band, and (local + global) the tiles
    // holding a global key, or every tile when a row of this tile is global.  Uniform over the CTA.
    auto visit = [&](int kt) -> bool {
        const long j0 = (long)kt * KT32;
        if (j0 <= t_hi && j0 + KT32 - 1 >= t_lo) return true;
        if (!lg) return false;
        if (any_g_row) return true;
        for (int u = 0; u < KT32 && j0 + u < p.S; ++u)
            if (p.is_global[j0 + u]) return true;
        return false;
    };
    auto next_tile = [&](int kt) {
        for (++kt; kt < n_kt && !visit(kt); ++kt) {}
        return kt;
    };
    // K and V of a tile into registers (rows past the sequence as zeros), 16-byte loads
    float4 kr[LPT], vr[LPT];
    auto fetch = [&](int kt) {
        const long j0 = (long)kt * KT32;
#pragma unroll
        for (int u = 0; u < LPT; ++u) {
            const int e = tid + u * F32_THREADS, kk = e / (D / 4), c4 = e - kk * (D / 4);
            kr[u] = vr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kt < n_kt && j0 + kk < p.S) {
                kr[u] = reinterpret_cast<const float4*>(Kh + (j0 + kk) * D)[c4];
                vr[u] = reinterpret_cast<const float4*>(Vh + (j0 + kk) * D)[c4];
            }
        }
    };

    float m = -INFINITY, l = 0.f, acc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) acc[c] = 0.f;
    int kt = visit(0) ? 0 : next_tile(0);
    if (kt < n_kt) fetch(kt);
    while (kt < n_kt) {
        const long j0 = (long)kt * KT32;
#pragma unroll
        for (int u = 0; u < LPT; ++u) {
            const int e = tid + u * F32_THREADS, kk = e / (D / 4), c4 = e - kk * (D / 4);
            *reinterpret_cast<float4*>(&sm.k[kk][4 * c4]) = kr[u];
            *reinterpret_cast<float4*>(&sm.v[kk][4 * c4]) = vr[u];
        }
        __syncthreads();
        const int kn = next_tile(kt);
        if (kn < n_kt) fetch(kn);  // the next tile's loads fly while this one is computed
        // scores of this thread's keys g, g + TPR
        float sc[KPT];
#pragma unroll
        for (int u = 0; u < KPT; ++u) sc[u] = 0.f;
#pragma unroll 16
        for (int c = 0; c < D; ++c) {
            const float qv = sm.q[r][c];
#pragma unroll
            for (int u = 0; u < KPT; ++u) sc[u] = fmaf(qv, sm.k[g + TPR * u][c], sc[u]);
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < KPT; ++u) {
            const long j = j0 + g + TPR * u;
            bool ok = j < p.S && j >= lo && j <= hi;
            if (lg && !ok && j < p.S && row_valid) ok = p.is_global[j];
            float s = sc[u] * p.scale;
            if (p.alibi) s -= slope * fabsf((float)(i - j));  // additive bias -m_a |i - j|
            sc[u] = ok ? s : -INFINITY;
            tmax = fmaxf(tmax, sc[u]);
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        const float m_new = fmaxf(m, tmax);
        const float ref = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = expf(m - ref);  // 0 while m is -inf
        float psum = 0.f;
#pragma unroll
        for (int u = 0; u < KPT; ++u) {
            const float pe = expf(sc[u] - ref);  // 0 where masked
            sm.p[r][g + TPR * u] = pe;
            psum += pe;
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l = l * alpha + psum;
        m = m_new;
        __syncwarp();  // the row's P, written by its lanes (one warp holds two rows), before they read it
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] *= alpha;
#pragma unroll 8
        for (int kk = 0; kk < KT32; ++kk) {
            const float pk = sm.p[r][kk];
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[c] = fmaf(pk, sm.v[kk][g + TPR * c], acc[c]);
        }
        __syncthreads();  // every thread is done with this K, V and P before the next tile overwrites them
        kt = kn;
    }

    if (row_valid) {
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        float* o = p.o + (bh * p.S + i) * D;
#pragma unroll
        for (int c = 0; c < CPT; ++c) o[g + TPR * c] = acc[c] * inv_l;
        if (p.lse && g == 0) p.lse[bh * p.S + i] = l > 0.f ? m + logf(l) : -INFINITY;
    }
}

// Evaluates the FMA-pipe exp2 (exp2_poly2, kept for the exponential-offload experiments) elementwise, for its test.
__global__ void exp2_selftest_kernel(const float* x, float* y, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const float2 v = make_float2(x[i], i + 1 < n ? x[i + 1] : 0.f);
    const float2 r = ptx::exp2_poly2(v);
    y[i] = r.x;
    if (i + 1 < n) y[i + 1] = r.y;
}

}  // namespace

cudaError_t launch_exp2_selftest(const float* x, float* y, int n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int pairs = (n + 1) / 2;
    exp2_selftest_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y, n);
    return cudaGetLastError();
}

cudaError_t launch_f32_forward(const F32Params& p, int d, cudaStream_t stream) {
    const long n_blocks = (long)p.B * p.Hq * ((p.S + QT - 1) / QT);
    if (n_blocks > 0x7fffffffL) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)n_blocks;
    if (d == 128) attn_fwd_f32_kernel<128><<<grid, F32_THREADS, 0, stream>>>(p);
    else if (d == 64) attn_fwd_f32_kernel<64><<<grid, F32_THREADS, 0, stream>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace attn
