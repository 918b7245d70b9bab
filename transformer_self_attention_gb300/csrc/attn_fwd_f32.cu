// fp32 attention forward on CUDA cores, and the self-test of the FMA-pipe exp2.
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

}  // namespace attn
