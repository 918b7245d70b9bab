// Kernel parameter blocks and launchers shared by the host code and the CUDA
// translation units of the library.  Internal; the public ABI is attn.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Parameters of the tensor-core (tcgen05) forward kernel.  Passed by value
// as a __grid_constant__ so the TMA descriptors live in parameter space.
struct TcParams {
    CUtensorMap tm_q;    // Q  [B*Hq,  S, d] bf16, box {64, 128, 1}, 128B swizzle
    CUtensorMap tm_k;    // K  [B*Hkv, S, d], box {64, tc_kv_box_rows(d), 1}
    CUtensorMap tm_v;    // V  [B*Hkv, S, d], box {64, tc_kv_box_rows(d), 1}
    CUtensorMap tm_o;    // O  [B*Hq,  S, d] (TMA store)
    const int4* work;    // 4 int4 per work item (attn.h schedule layout)
    int item_offset;     // first work item of this launch
    int S, Hq, Hkv, group;
    int kind, window;
    float scale_log2;    // scale * log2(e)
    const int* globals;  // sorted global positions (device)
    int n_global;
    const unsigned* global_bits;  // 4 words per 128-position tile (key tiles and query tiles alike)
    // per query tile {g_lo, g_hi}: the globals outside its band of key tiles are G[0, g_lo) and
    // G[g_hi, n_global) (local + global)
    const int2* gsplit;
    // local + global: the bf16 bits of Q, K, V, from which the producer warp gathers the global
    // rows (query rows of the global-row items, keys and values of the gathered key tiles)
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    void* o;             // O base (direct row stores)
    float* lse;          // may be null
    int* err;            // device error word
    long long watchdog_ns;
    int withhold_v;      // test hook: producer never loads V
    // global-row items split into key chunks (n_chunks > 1): partial results per chunk, and per
    // (batch-head, global-row tile) a counter of the chunks that have finished; the last chunk to
    // finish merges them and puts the counter back to 0
    float* part_o;       // [B*Hq, n_global, n_chunks, d] fp32, each normalised by its own sum
    float* part_lse;     // [B*Hq, n_global, n_chunks]
    int n_chunks;
    unsigned* counters;  // [B*Hq*n_gtiles]
    int n_gtiles;        // global-row tiles per (batch, head): ceil(n_global / 128)
    const float* alibi;  // [Hq] slopes of the additive bias -m_a |i - j| (device), or null
    int fp8;             // Q, K, V are E4M3 (scale_log2 includes their descales)
    float o_scale;       // factor on O at the end (the V descale for E4M3 inputs, else 1)
    // additive bias matrix (bf16 [bias_Bb, bias_Hb, S, bias_ld], device), or null; tm_bias
    // covers it as {bias_ld, S, bias_Bb * bias_Hb} with box {128, 128, 1} (L2 prefetches)
    CUtensorMap tm_bias;
    const uint16_t* bias;
    int bias_Bb, bias_Hb;
    long bias_ld;
};

// Rows of the box of the forward's K and V tensor maps (tm_k, tm_v): 64 at d = 64, where the
// tensor-core kernel may take 64-key tiles (a 128-key tile is then two copies), 128 otherwise.
constexpr unsigned tc_kv_box_rows(int d) { return d == 64 ? 64u : 128u; }

// Parameters of the fp32 CUDA-core kernel.
struct F32Params {
    const float* q; const float* k; const float* v;
    float* o; float* lse;
    int B, Hq, Hkv, S, group;
    int kind, window;
    float scale;
    const int* globals; int n_global;
    const unsigned char* is_global;  // [S] flags (local + global only)
    const float* alibi;  // [Hq] slopes of the additive bias -m_a |i - j| (device), or null
};

// Decode / key-value-cache attention (attn_decode.cu).  A persistent grid of n_cta
// CTAs shares the key tiles of all (sequence, kv head) units in one linear order:
// unit (b, g) covers indices [Hkv * tile_prefix[b] + g * n_b, ... + n_b) with
// n_b = tile_prefix[b+1] - tile_prefix[b], and CTA k takes indices
// [k * T / n_cta, (k+1) * T / n_cta), T = Hkv * tile_prefix[B].  A CTA processes the
// query rows of a kv head's group (group * S_q rows, padded to NP columns).
constexpr int kDecodeMaxBatch = 1024;
constexpr int kDecodeMaxCta = 512;  // the persistent grid is min(CTAs per SM x multiprocessors, this, tiles)
struct DecodeParams {
    CUtensorMap tm_q;    // Q as 2-D [B*Hq*S_q, d] bf16, box {64, NP}, 128B swizzle
    CUtensorMap tm_k;    // K cache [B*Hkv, S_cap, d], box {64, 128, 1}
    CUtensorMap tm_v;    // V cache [B*Hkv, S_cap, d]
    void* o;             // O [B, Hq, S_q, d] bf16
    float* lse;          // [B, Hq, S_q], may be null
    float* part_o;       // units split over CTAs: [2 * n_cta][NP][d] fp32 partial O (normalised by its own sum)
    float* part_lse;     // [2 * n_cta][NP]
    unsigned* counters;  // [B*Hkv] arrival counters of split units (wrap to 0)
    int* err;
    long long watchdog_ns;
    int B, Hq, Hkv, group, S_q, S_cap, rows;  // rows = group * S_q
    int kind, window;
    float scale_log2;
    int n_cta;
    long long total_tiles;                   // T
    const float* alibi;                      // [Hq] slopes of the bias -m_a |t - j| (device), or null
    int defer_merge;                         // split units: leave the partials to the merge kernel
    int len[kDecodeMaxBatch];                // cache length of each sequence
    int tile_prefix[kDecodeMaxBatch + 1];    // key tiles of the sequences before b (per kv head)
    long long share[kDecodeMaxCta + 1];      // CTA k takes the list indices [share[k], share[k+1])
};

cudaError_t launch_decode(const DecodeParams& p, int d, int np, cudaStream_t stream);

// Merge of the units split over several CTAs, as a kernel of its own: one warp per packed row.
constexpr int kDecodeMaxSplit = 512;
struct DecodeMergeParams {
    const float* part_o;    // the decode kernel's partial slots
    const float* part_lse;
    void* o;                // O [B, Hq, S_q, d] bf16
    float* lse;             // [B, Hq, S_q], may be null
    int Hq, group, S_q, rows, np, n_split;
    int4 list[kDecodeMaxSplit];  // split unit u: {b, g, k0, 2 * nseg + (unit starts CTA k0's share)}
};
cudaError_t launch_decode_merge(const DecodeMergeParams& p, int d, cudaStream_t stream);

// Backward pass (attn_bwd.cu): a pre-pass (D = dO . O and LSE in log2 units, padded to
// S_pad rows per head), the dQ kernel (one CTA per forward work item) and the dK/dV kernel
// (one CTA per key tile and kv head).
struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;  // bf16 inputs, box {64, 128, 1}
    CUtensorMap tm_dq, tm_dk, tm_dv;      // bf16 outputs (TMA stores)
    const int4* work;     // dQ: the forward items (2 int4 each); dK/dV: the key-tile items
    int n_items;          // dK/dV: key-tile items per (batch, kv head)
    int S, S_pad, Hq, Hkv, group, kind, window;
    float scale_log2;     // scale * log2(e)
    float scale;
    const float* nlse2;   // [B*Hq, S_pad]: -LSE * log2(e); -inf past S
    const float* nd;      // [B*Hq, S_pad]: -D = -dO . O; 0 past S
    const float* alibi;   // [Hq] ALiBi slopes of the forward (device), or null
    const uint16_t* bias; // the forward's bias matrix (bf16 bits [bias_Bb, bias_Hb, S, bias_ld]), or null
    int bias_Bb, bias_Hb;
    long bias_ld;
    // local + global: the per-tile lists of partner tiles (entries t | kListFull when every pair
    // of the two tiles is allowed; the items index them) and the global positions as 4 words of
    // bits per 128-position tile; null otherwise
    const int* list;
    const unsigned* gbits;
    int* err;
    long long watchdog_ns;
};
constexpr int kListFull = ATTN_LIST_FULL;  // the FULL flag of a list entry (the tile index is below it)
struct BwdPrepParams {
    const uint16_t* o; const uint16_t* dout;  // bf16 bits [B*Hq, S, d]
    const float* lse;                          // [B*Hq, S] (natural log)
    float* nlse2; float* nd;                   // [B*Hq, S_pad]
    int BHq, S, S_pad, d;
};
cudaError_t launch_bwd_prep(const BwdPrepParams& p, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdParams& p, int d, int n_items, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, int n_ctas, cudaStream_t stream);

cudaError_t launch_tc_forward(const TcParams& p, int d, int n_items, cudaStream_t stream);
cudaError_t launch_f32_forward(const F32Params& p, int d, cudaStream_t stream);
cudaError_t launch_exp2_selftest(const float* x, float* y, int n, cudaStream_t stream);

}  // namespace attn
