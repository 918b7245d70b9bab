// fp32 attention forward on CUDA cores, and the gather of global-token rows.
//
// The fp32 path keeps full fp32 inputs and arithmetic (TF32 tensor cores
// would round the inputs to 10 mantissa bits).  One warp owns one query row:
// the lanes split the head dimension, a warp reduction forms each score, and
// the running max / sum recurrence of the online softmax ("Transformer 演进与变体"
// (ai.icyfenix.cn), section Flash Attention, 在线 Softmax) is applied key by key.
// Keys are visited only where the mask allows them: the row's window interval,
// then (local + global) the global keys outside it, or every key for a
// global row ("Transformer 演进与变体", section 稀疏注意力).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn.h"
#include "kernels.h"
#include "sm103_ptx.h"

namespace attn {
namespace {

constexpr int ROWS_PER_BLOCK = 8;  // one warp per row

template <int D>
__global__ void __launch_bounds__(32 * ROWS_PER_BLOCK) attn_fwd_f32_kernel(F32Params p) {
    constexpr int E = D / 32;  // elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long row = (long)blockIdx.x * ROWS_PER_BLOCK + warp;
    const long n_rows = (long)p.B * p.Hq * p.S;
    if (row >= n_rows) return;
    const long bh = row / p.S;
    const long i = row - bh * p.S;
    const long b = bh / p.Hq, a = bh - b * p.Hq;
    const long bkv = b * p.Hkv + a / p.group;  // g(a) = a / (Hq / Hkv)
    const float* q = p.q + row * D;
    const float* Kh = p.k + bkv * (long)p.S * D;
    const float* Vh = p.v + bkv * (long)p.S * D;

    float qv[E], acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) { qv[e] = q[lane + 32 * e]; acc[e] = 0.f; }
    const float slope = p.alibi ? p.alibi[a] : 0.f;
    float m = -INFINITY, l = 0.f;

    auto visit = [&](long j) {
        const float* k = Kh + j * D;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qv[e], k[lane + 32 * e], dot);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        float s = dot * p.scale;
        if (p.alibi) s -= slope * fabsf((float)(i - j));  // additive bias -m_a |i - j|
        const float m_new = fmaxf(m, s);
        const float c = expf(m - m_new);  // 0 on the first key
        const float e_s = expf(s - m_new);
        l = l * c + e_s;
        const float* v = Vh + j * D;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(acc[e], c, e_s * v[lane + 32 * e]);
        m = m_new;
    };

    const bool lg = p.kind == ATTN_MASK_LOCAL_GLOBAL;
    const bool g_row = lg && p.n_global > 0 && p.is_global[i];
    long lo = 0, hi = p.S - 1;
    if (g_row) {
        // a global row sees every key
    } else if (p.kind == ATTN_MASK_CAUSAL) {
        hi = i;
    } else if (p.kind == ATTN_MASK_CAUSAL_SLIDING) {
        lo = i - p.window > 0 ? i - p.window : 0;
        hi = i;
    } else if (p.kind == ATTN_MASK_SLIDING || lg) {
        lo = i - p.window > 0 ? i - p.window : 0;
        hi = i + p.window < p.S - 1 ? i + p.window : p.S - 1;
    }
    for (long j = lo; j <= hi; ++j) visit(j);
    if (lg && !g_row)
        for (int t = 0; t < p.n_global; ++t) {
            const long j = p.globals[t];
            if (j < lo || j > hi) visit(j);
        }

    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    float* o = p.o + row * D;
#pragma unroll
    for (int e = 0; e < E; ++e) o[lane + 32 * e] = acc[e] * inv_l;
    if (p.lse && lane == 0) p.lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
}

// Copy rows globals[r] of Q (per query head) and of K, V (per kv head) into
// dense [heads, n_global, d] scratch tensors.  blockIdx.x = r, blockIdx.y =
// head slot over Q heads then K heads then V heads; 16-byte vectors.
__global__ void gather_globals_kernel(GatherParams p) {
    const int r = blockIdx.x;
    int slot = blockIdx.y;
    const uint16_t* src;
    uint16_t* dst;
    long head;
    if (slot < p.BHq) { src = p.q; dst = p.qg; head = slot; }
    else if ((slot -= p.BHq) < p.BHkv) { src = p.k; dst = p.kg; head = slot; }
    else { slot -= p.BHkv; src = p.v; dst = p.vg; head = slot; }
    const long pos = p.globals[r];
    const uint4* s4 = reinterpret_cast<const uint4*>(src + (head * p.S + pos) * p.d);
    uint4* d4 = reinterpret_cast<uint4*>(dst + (head * p.n_global + r) * p.d);
    for (int t = threadIdx.x; t < p.d / 8; t += blockDim.x) d4[t] = s4[t];
}

// Combines the key chunks of the global-row pass.  One warp per (head, global
// row).  Chunk c holds O_c (its own softmax-weighted average) and
// LSE_c = ln of its sum of exponentials, so the whole row is
//   O = sum_c e^(LSE_c - M) O_c / sum_c e^(LSE_c - M),  LSE = M + ln sum_c e^(LSE_c - M)
// with M = max_c LSE_c: the same softmax normalisation, applied across chunks.
// Lanes split the chunks for M and the weights (warp reductions), then split d for the
// weighted sum, each weight broadcast from the lane that computed it; the partial-O loads
// of eight chunks are issued before their multiply-adds (the merge is latency-bound).
__global__ void merge_global_rows_kernel(MergeParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long row = (long)blockIdx.x * (blockDim.x >> 5) + warp;
    if (row >= (long)p.BHq * p.n_global) return;
    const long bh = row / p.n_global;
    const int gr = (int)(row - bh * p.n_global);
    const float* lse_c = p.part_lse + row * p.n_chunks;
    float M = -INFINITY;
    for (int c = lane; c < p.n_chunks; c += 32) M = fmaxf(M, lse_c[c]);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
    float W = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // d <= 128: 4 elements per lane
    const int nd = p.d / 32;
    for (int c0 = 0; c0 < p.n_chunks; c0 += 32) {
        const int c = c0 + lane;
        const float wl = c < p.n_chunks ? expf(lse_c[c] - M) : 0.f;  // this lane's chunk weight
        W += wl;
        const int n_here = min(32, p.n_chunks - c0);
        const float* ob = p.part_o + (row * p.n_chunks + c0) * p.d;
        for (int j0 = 0; j0 < n_here; j0 += 8) {
            float v[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v[j][e] = (j0 + j < n_here && e < nd) ? ob[(long)(j0 + j) * p.d + lane + 32 * e] : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float wc = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);  // 0 past the last chunk
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = fmaf(wc, v[j][e], acc[e]);
            }
        }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) W += __shfl_xor_sync(0xffffffffu, W, s);
    const long pos = p.globals[gr];
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.o) + (bh * p.S + pos) * p.d;
    for (int e = 0; e < nd; ++e) o[lane + 32 * e] = __float2bfloat16_rn(acc[e] / W);
    if (p.lse && lane == 0) p.lse[bh * p.S + pos] = M + logf(W);
}

// Evaluates the softmax warps' FMA-pipe exp2 (exp2_poly2) elementwise, for its test.
__global__ void exp2_selftest_kernel(const float* x, float* y, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const float2 v = make_float2(x[i], i + 1 < n ? x[i + 1] : 0.f);
    const float2 r = ptx::exp2_poly2(v);
    y[i] = r.x;
    if (i + 1 < n) y[i + 1] = r.y;
}

}  // namespace

cudaError_t launch_merge_global_rows(const MergeParams& p, cudaStream_t stream) {
    const long rows = (long)p.BHq * p.n_global;
    if (rows <= 0) return cudaSuccess;
    merge_global_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_exp2_selftest(const float* x, float* y, int n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int pairs = (n + 1) / 2;
    exp2_selftest_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y, n);
    return cudaGetLastError();
}

cudaError_t launch_f32_forward(const F32Params& p, int d, cudaStream_t stream) {
    const long n_rows = (long)p.B * p.Hq * p.S;
    const unsigned grid = (unsigned)((n_rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK);
    if (d == 128) attn_fwd_f32_kernel<128><<<grid, 32 * ROWS_PER_BLOCK, 0, stream>>>(p);
    else if (d == 64) attn_fwd_f32_kernel<64><<<grid, 32 * ROWS_PER_BLOCK, 0, stream>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_gather_globals(const GatherParams& p, cudaStream_t stream) {
    if (p.n_global <= 0) return cudaSuccess;
    dim3 grid((unsigned)p.n_global, (unsigned)(p.BHq + 2 * p.BHkv));
    gather_globals_kernel<<<grid, 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
