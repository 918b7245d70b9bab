// Host implementation of the decode / key-value-cache entry points of include/attn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <new>

#include "attn.h"
#include "kernels.h"
#include "schedule.h"

namespace attn {
int decode_ctas_per_sm(int d, int np);  // attn_decode.cu
}

struct attn_decode_plan {
    int B = 0, Hq = 0, Hkv = 0, S_q = 0, S_cap = 0, d = 0, np = 0;
    int ctas_per_sm = 1;  // CTAs of the persistent grid per multiprocessor
    int kind = 0, window = 0;
    float scale = 0.f;
    int n_sm = 0;
    int grid_limit = 0;  // test hook: 0 = one CTA per multiprocessor
    int merge_mode = 0;  // split units: 0 auto, 1 merged in the decode kernel, 2 by the merge kernel
    int last_launches = 0;  // kernels the last attn_decode_forward launched
    size_t part_slots = 0;
    int* d_err = nullptr;
    unsigned* d_counters = nullptr;
    float* d_part = nullptr;
    float* d_alibi = nullptr;  // ALiBi slopes [Hq] (attn_decode_set_alibi), or null
    const void* last_q = nullptr;
    const void* last_k = nullptr;
    const void* last_v = nullptr;
    attn::DecodeParams p{};
    attn::DecodeMergeParams mp{};
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// bf16 map, 128-byte swizzle, box {64, box_rows[, 1]}; rank 2 ([rows, d]) or 3 ([heads, rows, d]).
bool encode(CUtensorMap* map, const void* base, int d, long rows, long heads, unsigned box_rows, int rank) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool decode_kind(attn_mask_kind k) {
    return k == ATTN_MASK_FULL || k == ATTN_MASK_CAUSAL || k == ATTN_MASK_CAUSAL_SLIDING;
}

attn_status validate_decode(int B, int Hq, int Hkv, int S_q, int S_cap, attn_mask_kind kind, int window) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || S_q < 1 || S_cap < 1 || S_cap > (1 << 24))
        return ATTN_ERR_INVALID_ARG;
    if ((int)kind < ATTN_MASK_FULL || (int)kind > ATTN_MASK_LOCAL_GLOBAL) return ATTN_ERR_INVALID_ARG;
    if (!decode_kind(kind)) return ATTN_ERR_UNSUPPORTED;
    if (kind == ATTN_MASK_CAUSAL_SLIDING && window < 0) return ATTN_ERR_INVALID_ARG;
    if (kind != ATTN_MASK_FULL && S_q > S_cap) return ATTN_ERR_INVALID_ARG;
    if (B > ATTN_DECODE_MAX_BATCH || (long)(Hq / Hkv) * S_q > ATTN_DECODE_MAX_ROWS) return ATTN_ERR_UNSUPPORTED;
    if ((long)B * Hq * S_q > (1L << 30) || (long)B * Hkv > (1L << 30)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

attn_status validate_lengths(int B, int S_q, int S_cap, attn_mask_kind kind, const int* lens) {
    if (!lens) return ATTN_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 1 || lens[b] > S_cap) return ATTN_ERR_INVALID_ARG;
        if (kind != ATTN_MASK_FULL && lens[b] < S_q) return ATTN_ERR_INVALID_ARG;
    }
    return ATTN_OK;
}

void free_decode(attn_decode_plan* h) {
    if (!h) return;
    if (h->d_err) cudaFree(h->d_err);
    if (h->d_counters) cudaFree(h->d_counters);
    if (h->d_part) cudaFree(h->d_part);
    if (h->d_alibi) cudaFree(h->d_alibi);
    delete h;
}

}  // namespace

extern "C" {

attn_status attn_decode_create(attn_decode_handle* out, int B, int Hq, int Hkv, int S_q, int S_cap, int d_k,
                               float scale, attn_mask_kind kind, int window) {
    if (!out) return ATTN_ERR_INVALID_ARG;
    *out = nullptr;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    attn_status vs = validate_decode(B, Hq, Hkv, S_q, S_cap, kind, window);
    if (vs != ATTN_OK) return vs;
    if (d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED;

    attn_decode_plan* h = new (std::nothrow) attn_decode_plan();
    if (!h) return ATTN_ERR_OOM;
    h->B = B; h->Hq = Hq; h->Hkv = Hkv; h->S_q = S_q; h->S_cap = S_cap; h->d = d_k;
    h->kind = kind; h->window = kind == ATTN_MASK_CAUSAL_SLIDING ? window : 0; h->scale = scale;
    const int rows = (Hq / Hkv) * S_q;
    h->np = rows <= 16 ? 16 : rows <= 32 ? 32 : 64;

    auto fail = [&](cudaError_t err) {
        free_decode(h);
        return err == cudaErrorMemoryAllocation ? ATTN_ERR_OOM : ATTN_ERR_CUDA;
    };
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(e);
    // two partial-result slots per CTA of the persistent grid (its first and last stretch)
    h->ctas_per_sm = attn::decode_ctas_per_sm(d_k, h->np);
    h->part_slots = 2 * (size_t)h->n_sm * h->ctas_per_sm;
    if ((e = cudaMalloc(reinterpret_cast<void**>(&h->d_err), sizeof(int))) != cudaSuccess) return fail(e);
    if ((e = cudaMemset(h->d_err, 0, sizeof(int))) != cudaSuccess) return fail(e);
    if ((e = cudaMalloc(reinterpret_cast<void**>(&h->d_counters), sizeof(unsigned) * B * Hkv)) != cudaSuccess)
        return fail(e);
    if ((e = cudaMemset(h->d_counters, 0, sizeof(unsigned) * B * Hkv)) != cudaSuccess) return fail(e);
    if ((e = cudaMalloc(reinterpret_cast<void**>(&h->d_part), h->part_slots * h->np * (d_k + 1) * sizeof(float))) !=
        cudaSuccess)
        return fail(e);

    attn::DecodeParams& p = h->p;
    p.part_o = h->d_part;
    p.part_lse = h->d_part + h->part_slots * h->np * d_k;
    p.counters = h->d_counters;
    p.err = h->d_err;
    p.watchdog_ns = 2000000000LL;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.group = Hq / Hkv; p.S_q = S_q; p.S_cap = S_cap; p.rows = rows;
    p.kind = kind; p.window = h->window;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    *out = h;
    return ATTN_OK;
}

attn_status attn_decode_forward(attn_decode_handle h, const void* Q, const void* K, const void* V,
                                const int* cache_len, void* O, float* LSE, void* stream) {
    if (!h || !Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u))
        return ATTN_ERR_INVALID_ARG;
    attn_status vs = validate_lengths(h->B, h->S_q, h->S_cap, (attn_mask_kind)h->kind, cache_len);
    if (vs != ATTN_OK) return vs;
    attn::DecodeParams& p = h->p;
    if (Q != h->last_q) {
        if (!encode(&p.tm_q, Q, h->d, (long)h->B * h->Hq * h->S_q, 1, (unsigned)h->np, 2)) return ATTN_ERR_CUDA;
        h->last_q = Q;
    }
    if (K != h->last_k) {
        if (!encode(&p.tm_k, K, h->d, h->S_cap, (long)h->B * h->Hkv, ATTN_TILE, 3)) return ATTN_ERR_CUDA;
        h->last_k = K;
    }
    if (V != h->last_v) {
        if (!encode(&p.tm_v, V, h->d, h->S_cap, (long)h->B * h->Hkv, ATTN_TILE, 3)) return ATTN_ERR_CUDA;
        h->last_v = V;
    }
    attn::DecodeSchedule sched;
    const int grid = h->n_sm * h->ctas_per_sm;
    const int ctas = std::min(h->grid_limit > 0 ? std::min(h->grid_limit, grid) : grid, attn::kDecodeMaxCta);
    attn::build_decode_schedule(h->B, h->Hkv, h->S_q, h->kind, h->window, cache_len, ctas, &sched);
    if (2 * (size_t)sched.n_cta > h->part_slots) return ATTN_ERR_UNSUPPORTED;  // cannot happen: n_cta <= grid
    for (int b = 0; b < h->B; ++b) p.len[b] = cache_len[b];
    for (int b = 0; b <= h->B; ++b) p.tile_prefix[b] = sched.tile_prefix[b];
    for (int k = 0; k <= sched.n_cta; ++k) p.share[k] = sched.share[k];
    p.n_cta = sched.n_cta;
    p.total_tiles = sched.total_tiles;
    p.o = O;
    p.lse = LSE;
    // Units split over several CTAs (CTA k takes the indices [share[k], share[k + 1])).  By
    // default their partial results are combined by the merge kernel, launched as a dependent
    // of the decode kernel so that its launch overlaps the decode kernel's tail: a merge by the
    // last CTA to finish a part sits at the end of that CTA's share (a serial tail of L2 round
    // trips the share weights do not see).
    attn::DecodeMergeParams& mp = h->mp;
    const std::vector<long long>& share = sched.share;
    auto share_of = [&](long long i) {  // the CTA whose share holds index i
        return (int)(std::upper_bound(share.begin(), share.end() - 1, i) - share.begin()) - 1;
    };
    mp.n_split = 0;
    bool overflow = false;
    for (int b = 0; b < h->B; ++b) {
        const int n_unit = sched.tile_prefix[b + 1] - sched.tile_prefix[b];
        for (int g = 0; g < h->Hkv && n_unit > 0; ++g) {
            const long long ub = (long long)h->Hkv * sched.tile_prefix[b] + (long long)g * n_unit;
            const int k0 = share_of(ub), k1 = share_of(ub + n_unit - 1);
            if (k1 == k0) continue;
            if (mp.n_split == attn::kDecodeMaxSplit) { overflow = true; continue; }
            const bool first = share[k0] == ub;
            mp.list[mp.n_split++] = make_int4(b, g, k0, 2 * (k1 - k0 + 1) + (first ? 1 : 0));
        }
    }
    const bool defer = !overflow && mp.n_split > 0 && h->merge_mode != 1;
    p.defer_merge = defer ? 1 : 0;
    cudaError_t e = attn::launch_decode(p, h->d, h->np, static_cast<cudaStream_t>(stream));
    h->last_launches = defer ? 2 : 1;
    if (e == cudaSuccess && defer) {
        mp.part_o = p.part_o;
        mp.part_lse = p.part_lse;
        mp.o = O;
        mp.lse = LSE;
        mp.Hq = h->Hq; mp.group = h->Hq / h->Hkv; mp.S_q = h->S_q; mp.rows = p.rows; mp.np = h->np;
        e = attn::launch_decode_merge(mp, h->d, static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_decode_poll_device_error(attn_decode_handle h, int* code) {
    if (!h || !code) return ATTN_ERR_INVALID_ARG;
    *code = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpy(code, h->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (*code != 0) {
        // an aborted CTA leaves its units' arrival counters part-way: start them again
        if (cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaMemset(h->d_counters, 0, sizeof(unsigned) * h->B * h->Hkv) != cudaSuccess) return ATTN_ERR_CUDA;
    }
    return *code ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
}

attn_status attn_decode_set_alibi(attn_decode_handle h, const float* slopes) {
    if (!h) return ATTN_ERR_INVALID_ARG;
    if (!slopes) {
        if (h->d_alibi) cudaFree(h->d_alibi);
        h->d_alibi = nullptr;
        h->p.alibi = nullptr;
        return ATTN_OK;
    }
    for (int a = 0; a < h->Hq; ++a)
        if (!std::isfinite(slopes[a])) return ATTN_ERR_INVALID_ARG;
    if (!h->d_alibi) {
        cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&h->d_alibi), sizeof(float) * h->Hq);
        if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? ATTN_ERR_OOM : ATTN_ERR_CUDA;
    }
    if (cudaMemcpy(h->d_alibi, slopes, sizeof(float) * h->Hq, cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_ERR_CUDA;
    h->p.alibi = h->d_alibi;
    return ATTN_OK;
}

attn_status attn_decode_launch_count(attn_decode_handle h, int* n) {
    if (!h || !n) return ATTN_ERR_INVALID_ARG;
    *n = h->last_launches;
    return ATTN_OK;
}

attn_status attn_decode_set_merge_mode(attn_decode_handle h, int mode) {
    if (!h || mode < 0 || mode > 2) return ATTN_ERR_INVALID_ARG;
    h->merge_mode = mode;
    return ATTN_OK;
}

attn_status attn_decode_set_grid_limit(attn_decode_handle h, int max_ctas) {
    if (!h || max_ctas < 1) return ATTN_ERR_INVALID_ARG;
    h->grid_limit = max_ctas;
    return ATTN_OK;
}

attn_status attn_decode_destroy(attn_decode_handle h) {
    if (!h) return ATTN_OK;
    cudaError_t e = cudaDeviceSynchronize();
    free_decode(h);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_decode_schedule_host(int B, int Hkv, int S_q, int S_cap, attn_mask_kind kind, int window,
                                      const int* cache_len, int n_sm, int* n_cta, int* tile_prefix,
                                      long long* share) {
    if (!n_cta || !tile_prefix || !share || n_sm < 1) return ATTN_ERR_INVALID_ARG;
    attn_status vs = validate_decode(B, Hkv, Hkv, S_q, S_cap, kind, window);
    if (vs != ATTN_OK) return vs;
    vs = validate_lengths(B, S_q, S_cap, kind, cache_len);
    if (vs != ATTN_OK) return vs;
    attn::DecodeSchedule sched;
    attn::build_decode_schedule(B, Hkv, S_q, kind, kind == ATTN_MASK_CAUSAL_SLIDING ? window : 0, cache_len,
                                std::min(n_sm, attn::kDecodeMaxCta), &sched);
    *n_cta = sched.n_cta;
    for (int b = 0; b <= B; ++b) tile_prefix[b] = sched.tile_prefix[b];
    for (int k = 0; k <= sched.n_cta; ++k) share[k] = sched.share[k];
    return ATTN_OK;
}

}  // extern "C"
