// Host implementation of the C ABI declared in include/attn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "attn.h"
#include "device_once.h"
#include "kernels.h"
#include "schedule.h"

struct attn_plan {
    int B = 0, Hq = 0, Hkv = 0, S = 0, d = 0;
    attn_dtype dtype = ATTN_BF16;
    float scale = 0.f;
    int kind = 0, window = 0;
    std::vector<int> globals;
    attn::Schedule sched;
    // device buffers owned by the handle
    int4* d_work = nullptr;
    int* d_globals = nullptr;
    unsigned* d_gbits = nullptr;
    int* d_gsplit = nullptr;
    unsigned char* d_isg = nullptr;
    int* d_err = nullptr;
    float* d_part = nullptr;  // partial results of the chunked global-row items
    unsigned* d_counters = nullptr;  // their arrival counters (each returns to 0 when its tile is merged)
    float* d_alibi = nullptr;  // ALiBi slopes [Hq] (attn_set_alibi), or null
    // backward scratch (first attn_backward call)
    float* d_lse2 = nullptr;   // [B*Hq, S_pad]
    float* d_dvec = nullptr;   // [B*Hq, S_pad]
    int4* d_kvwork = nullptr;  // key-tile items
    int4* d_dqwork = nullptr;  // forward items regrouped by kv head (dQ launch)
    int* d_bwdlist = nullptr;  // local + global: the per-tile lists of partner tiles
    int n_kv_items = 0;
    int n_dq_items = 0;
    const void* last_bwd[7] = {};
    attn::BwdParams bp{};
    // tensor maps of the last pointers seen (re-encoded when they change)
    const void* last_q = nullptr;
    const void* last_k = nullptr;
    const void* last_v = nullptr;
    const void* last_o = nullptr;
    attn::TcParams tp{};
    bool debug = false;
};

namespace attn {
DeviceOnce& device_once() {
    static DeviceOnce registry;
    return registry;
}
}  // namespace attn

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 3-D bf16 map over [heads, rows, d] (d fastest), box {64, box_rows, 1}, 128-byte
// swizzle; rows past `rows` read as zeros and are not written by stores.
bool encode_map(CUtensorMap* map, const void* base, int d, long rows, long heads, unsigned box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same for E4M3 tensors (bytes): box {128, box_rows, 1}, one 128-byte swizzled row.
bool encode_map_e4m3(CUtensorMap* map, const void* base, int d, long rows, long heads, unsigned box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)rows * d};
    // rows of d bytes: one 128-byte swizzled block at d = 128, one 64-byte swizzled block at d = 64
    cuuint32_t box[3] = {(cuuint32_t)(d >= 128 ? 128 : 64), box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, d >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A bias matrix bf16 [planes, S, ld] for L2 prefetches of 128 x 128 boxes (no swizzle).
bool encode_map_bias(CUtensorMap* map, const void* base, long ld, long S, long planes) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)ld, (cuuint64_t)S, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)(S * ld * 2)};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

constexpr unsigned kTileRows = ATTN_TILE;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by attn_create and attn_schedule_host.
attn_status validate_shape(int B, int Hq, int Hkv, int S, attn_mask_kind kind, int window, const int* global_idx,
                           int n_global) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || S < 1 || S > (1 << 20)) return ATTN_ERR_INVALID_ARG;
    if ((int)kind < ATTN_MASK_FULL || (int)kind > ATTN_MASK_LOCAL_GLOBAL) return ATTN_ERR_INVALID_ARG;
    const bool windowed = kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_CAUSAL_SLIDING ||
                          kind == ATTN_MASK_LOCAL_GLOBAL;
    if (windowed && window < 0) return ATTN_ERR_INVALID_ARG;
    if (n_global < 0 || n_global > 4096) return ATTN_ERR_INVALID_ARG;
    if (n_global > 0 && (kind != ATTN_MASK_LOCAL_GLOBAL || !global_idx)) return ATTN_ERR_INVALID_ARG;
    for (int t = 0; t < n_global; ++t)
        if (global_idx[t] < 0 || global_idx[t] >= S) return ATTN_ERR_INVALID_ARG;
    if ((long)B * Hq > (1L << 30)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

std::vector<int> sorted_unique(const int* idx, int n) {
    std::vector<int> g(idx, idx + n);
    std::sort(g.begin(), g.end());
    g.erase(std::unique(g.begin(), g.end()), g.end());
    return g;
}

template <class T>
cudaError_t upload(T** dst, const T* src, size_t n) {
    if (n == 0) return cudaSuccess;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dst), n * sizeof(T));
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice);
}

void free_plan(attn_plan* h) {
    if (!h) return;
    void* bufs[] = {h->d_work, h->d_globals, h->d_gbits, h->d_gsplit, h->d_isg, h->d_err, h->d_part, h->d_counters,
                    h->d_alibi, h->d_lse2, h->d_dvec, h->d_kvwork, h->d_dqwork, h->d_bwdlist};
    for (void* b : bufs)
        if (b) cudaFree(b);
    delete h;
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
    switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device watchdog: a bounded wait ran out";
    case ATTN_ERR_OOM: return "out of memory";
    }
    return "unknown status";
}

attn_status attn_create(attn_handle* out, int B, int Hq, int Hkv, int S, int d_k, attn_dtype dtype, float scale,
                        attn_mask_kind kind, int window, const int* global_idx, int n_global) {
    if (!out) return ATTN_ERR_INVALID_ARG;
    *out = nullptr;
    if (dtype != ATTN_BF16 && dtype != ATTN_F32 && dtype != ATTN_FP8_E4M3) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    attn_status vs = validate_shape(B, Hq, Hkv, S, kind, window, global_idx, n_global);
    if (vs != ATTN_OK) return vs;
    if (d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED;
    const bool windowed = kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_CAUSAL_SLIDING ||
                          kind == ATTN_MASK_LOCAL_GLOBAL;

    attn_plan* h = new (std::nothrow) attn_plan();
    if (!h) return ATTN_ERR_OOM;
    h->B = B; h->Hq = Hq; h->Hkv = Hkv; h->S = S; h->d = d_k; h->dtype = dtype; h->scale = scale;
    h->kind = kind; h->window = windowed ? window : 0;
    h->globals = sorted_unique(global_idx, n_global);
    const char* dbg = std::getenv("ATTN_DEBUG");
    h->debug = dbg && dbg[0] == '1';

    attn::ScheduleInput in{B, Hq, Hkv, S, (int)kind, h->window, h->globals};
    attn_status st = attn::build_schedule(in, &h->sched);
    if (st != ATTN_OK) { free_plan(h); return st; }

    const int nG = (int)h->globals.size();
    cudaError_t e = cudaSuccess;
    auto fail = [&](cudaError_t err) {
        free_plan(h);
        return err == cudaErrorMemoryAllocation ? ATTN_ERR_OOM : ATTN_ERR_CUDA;
    };
    if ((e = cudaMalloc(reinterpret_cast<void**>(&h->d_err), sizeof(int))) != cudaSuccess) return fail(e);
    if ((e = cudaMemset(h->d_err, 0, sizeof(int))) != cudaSuccess) return fail(e);
    if (nG > 0) {
        if ((e = upload(&h->d_globals, h->globals.data(), h->globals.size())) != cudaSuccess) return fail(e);
        std::vector<unsigned char> isg(S, 0);
        for (int g : h->globals) isg[g] = 1;
        if ((e = upload(&h->d_isg, isg.data(), isg.size())) != cudaSuccess) return fail(e);
    }
    if (dtype == ATTN_BF16 || dtype == ATTN_FP8_E4M3) {
        if ((e = upload(reinterpret_cast<int**>(&h->d_work), h->sched.items.data(), h->sched.items.size())) !=
            cudaSuccess)
            return fail(e);
        if ((e = upload(&h->d_gbits, h->sched.global_bits.data(), h->sched.global_bits.size())) != cudaSuccess)
            return fail(e);
        if ((e = upload(&h->d_gsplit, h->sched.gsplit.data(), h->sched.gsplit.size())) != cudaSuccess)
            return fail(e);
        attn::TcParams& p = h->tp;
        p.n_gtiles = (nG + (int)kTileRows - 1) / (int)kTileRows;
        if (nG > 0 && h->sched.n_chunks > 1) {
            const size_t rows = (size_t)B * Hq * nG * h->sched.n_chunks;
            const size_t n_ctr = (size_t)B * Hq * p.n_gtiles;
            if ((e = cudaMalloc(reinterpret_cast<void**>(&h->d_part), rows * (d_k + 1) * sizeof(float))) !=
                    cudaSuccess ||
                (e = cudaMalloc(reinterpret_cast<void**>(&h->d_counters), n_ctr * sizeof(unsigned))) != cudaSuccess ||
                (e = cudaMemset(h->d_counters, 0, n_ctr * sizeof(unsigned))) != cudaSuccess)
                return fail(e);
        }
        p.work = h->d_work;
        p.S = S; p.Hq = Hq; p.Hkv = Hkv; p.group = Hq / Hkv;
        p.kind = kind; p.window = h->window;
        p.scale_log2 = (float)((double)scale * 1.4426950408889634);
        p.globals = h->d_globals;
        p.n_global = nG;
        p.global_bits = h->d_gbits;
        p.gsplit = reinterpret_cast<const int2*>(h->d_gsplit);
        p.err = h->d_err;
        p.watchdog_ns = 2000000000LL;
        p.withhold_v = 0;
        p.n_chunks = h->sched.n_chunks;
        p.fp8 = dtype == ATTN_FP8_E4M3;
        p.o_scale = 1.f;
        p.part_o = h->d_part;
        p.part_lse = h->d_part ? h->d_part + (size_t)B * Hq * nG * h->sched.n_chunks * d_k : nullptr;
        p.counters = h->d_counters;
    }
    *out = h;
    return ATTN_OK;
}

attn_status attn_forward(attn_handle h, const void* Q, const void* K, const void* V, void* O, float* LSE,
                         void* stream_ptr) {
    if (!h || !Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u))
        return ATTN_ERR_INVALID_ARG;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    cudaError_t e = cudaSuccess;
    const int nG = (int)h->globals.size();

    if (h->dtype == ATTN_F32) {
        attn::F32Params p{};
        p.q = static_cast<const float*>(Q); p.k = static_cast<const float*>(K); p.v = static_cast<const float*>(V);
        p.o = static_cast<float*>(O); p.lse = LSE;
        p.B = h->B; p.Hq = h->Hq; p.Hkv = h->Hkv; p.S = h->S; p.group = h->Hq / h->Hkv;
        p.kind = h->kind; p.window = h->window; p.scale = h->scale;
        p.globals = h->d_globals; p.n_global = nG; p.is_global = h->d_isg;
        p.alibi = h->d_alibi;
        e = attn::launch_f32_forward(p, h->d, stream);
    } else {
        attn::TcParams& p = h->tp;
        auto in_map = h->dtype == ATTN_FP8_E4M3 ? encode_map_e4m3 : encode_map;
        if (Q != h->last_q) {
            if (!in_map(&p.tm_q, Q, h->d, h->S, (long)h->B * h->Hq, kTileRows)) return ATTN_ERR_CUDA;
            h->last_q = Q;
        }
        if (K != h->last_k) {
            if (!in_map(&p.tm_k, K, h->d, h->S, (long)h->B * h->Hkv, attn::tc_kv_box_rows(h->d))) return ATTN_ERR_CUDA;
            h->last_k = K;
        }
        if (V != h->last_v) {
            if (!in_map(&p.tm_v, V, h->d, h->S, (long)h->B * h->Hkv, attn::tc_kv_box_rows(h->d))) return ATTN_ERR_CUDA;
            h->last_v = V;
        }
        if (O != h->last_o) {
            if (!encode_map(&p.tm_o, O, h->d, h->S, (long)h->B * h->Hq, kTileRows)) return ATTN_ERR_CUDA;
            h->last_o = O;
        }
        p.o = O;
        p.lse = LSE;
        p.q = static_cast<const uint16_t*>(Q);
        p.k = static_cast<const uint16_t*>(K);
        p.v = static_cast<const uint16_t*>(V);
        p.item_offset = 0;
        // one launch: the query-tile items, then (local + global) the global-row chunks
        e = attn::launch_tc_forward(p, h->d, h->sched.n_main + h->sched.n_grows, stream);
    }
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    if (h->debug) {
        int code = 0;
        return attn_poll_device_error(h, &code);
    }
    return ATTN_OK;
}

attn_status attn_destroy(attn_handle h) {
    if (!h) return ATTN_OK;
    cudaError_t e = cudaDeviceSynchronize();
    free_plan(h);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_schedule_host(int B, int Hq, int Hkv, int S, attn_mask_kind kind, int window,
                               const int* global_idx, int n_global, int* items, int cap, int* n_items,
                               int* n_first) {
    if (!n_items || !n_first || cap < 0 || (cap > 0 && !items)) return ATTN_ERR_INVALID_ARG;
    attn_status vs = validate_shape(B, Hq, Hkv, S, kind, window, global_idx, n_global);
    if (vs != ATTN_OK) return vs;
    const bool windowed = kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_CAUSAL_SLIDING ||
                          kind == ATTN_MASK_LOCAL_GLOBAL;
    attn::ScheduleInput in{B, Hq, Hkv, S, (int)kind, windowed ? window : 0, sorted_unique(global_idx, n_global)};
    attn::Schedule sched;
    attn_status st = attn::build_schedule(in, &sched);
    if (st != ATTN_OK) return st;
    const int n = (int)(sched.items.size() / ATTN_WORK_INTS);
    *n_items = n;
    *n_first = sched.n_main;
    if (cap == 0) return ATTN_OK;
    if (cap < n) return ATTN_ERR_INVALID_ARG;
    std::memcpy(items, sched.items.data(), sched.items.size() * sizeof(int));
    return ATTN_OK;
}

attn_status attn_kv_schedule_host(int S, attn_mask_kind kind, int window, int* items, int cap, int* n_items) {
    if (!n_items || cap < 0 || (cap > 0 && !items) || S < 1 || S > (1 << 20)) return ATTN_ERR_INVALID_ARG;
    if ((int)kind < ATTN_MASK_FULL || (int)kind > ATTN_MASK_LOCAL_GLOBAL) return ATTN_ERR_INVALID_ARG;
    const bool windowed = kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_CAUSAL_SLIDING;
    if (windowed && window < 0) return ATTN_ERR_INVALID_ARG;
    std::vector<int> v;
    attn_status st = attn::build_kv_schedule(S, kind, windowed ? window : 0, &v);
    if (st != ATTN_OK) return st;
    *n_items = (int)(v.size() / ATTN_WORK_INTS);
    if (cap == 0) return ATTN_OK;
    if (cap < *n_items) return ATTN_ERR_INVALID_ARG;
    std::memcpy(items, v.data(), v.size() * sizeof(int));
    return ATTN_OK;
}

attn_status attn_bwd_dq_schedule_host(int B, int Hq, int Hkv, int S, int d_k, attn_mask_kind kind, int window,
                                      int* items, int cap, int* n_items) {
    if (!n_items || cap < 0 || (cap > 0 && !items)) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || S < 1 || S > (1 << 20) || d_k < 1) return ATTN_ERR_INVALID_ARG;
    if ((int)kind < ATTN_MASK_FULL || (int)kind >= ATTN_MASK_LOCAL_GLOBAL) return ATTN_ERR_INVALID_ARG;
    const bool windowed = kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_CAUSAL_SLIDING;
    if (windowed && window < 0) return ATTN_ERR_INVALID_ARG;
    attn::ScheduleInput in{B, Hq, Hkv, S, (int)kind, windowed ? window : 0, {}};
    attn::Schedule sched;
    attn_status st = attn::build_schedule(in, &sched);
    if (st != ATTN_OK) return st;
    const std::vector<int> v = attn::order_dq_items(sched.items, sched.n_main, Hq, Hkv, attn::dq_kv_group(S, d_k));
    *n_items = sched.n_main;
    if (cap == 0) return ATTN_OK;
    if (cap < *n_items) return ATTN_ERR_INVALID_ARG;
    std::memcpy(items, v.data(), v.size() * sizeof(int));
    return ATTN_OK;
}

attn_status attn_bwd_lg_lists_host(int S, int window, const int* globals, int n_global, int* list, int cap,
                                   int* offsets, int* n_list) {
    if (!n_list || cap < 0 || (cap > 0 && (!list || !offsets)) || S < 1 || S > (1 << 20) || window < 0 ||
        n_global < 0 || (n_global > 0 && !globals))
        return ATTN_ERR_INVALID_ARG;
    for (int k = 0; k < n_global; ++k)
        if (globals[k] < 0 || globals[k] >= S) return ATTN_ERR_INVALID_ARG;
    std::vector<int> l, off;
    attn::build_lg_pair_lists(S, window, sorted_unique(globals, n_global), &l, &off);
    *n_list = (int)l.size();
    if (cap == 0) return ATTN_OK;
    if (cap < *n_list) return ATTN_ERR_INVALID_ARG;
    std::memcpy(list, l.data(), l.size() * sizeof(int));
    std::memcpy(offsets, off.data(), off.size() * sizeof(int));
    return ATTN_OK;
}

attn_status attn_poll_device_error(attn_handle h, int* code) {
    if (!h || !code) return ATTN_ERR_INVALID_ARG;
    *code = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpy(code, h->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (*code != 0 && cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    return *code ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
}

attn_status attn_selftest_exp2(const float* x, float* y, int n, void* stream) {
    if (!x || !y || n < 0) return ATTN_ERR_INVALID_ARG;
    return attn::launch_exp2_selftest(x, y, n, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                                 : ATTN_ERR_CUDA;
}

int attn_selftest_device_once(void) {
    attn::DeviceOnce reg;  // a private registry: the library's own is left untouched
    static const int kA = 0, kB = 0;
    const void* fa = &kA;
    const void* fb = &kB;
    int runs[4][2] = {};
    std::mutex mu;
    auto body = [&](int dev, int k) {
        return reg.run(dev, k ? fb : fa, 1024, [&] {
            std::lock_guard<std::mutex> lock(mu);
            ++runs[dev][k];
            return cudaSuccess;
        });
    };
    std::vector<std::thread> ts;
    for (int t = 0; t < 8; ++t)
        ts.emplace_back([&, t] {
            for (int r = 0; r < 50; ++r)
                for (int dev = 0; dev < 4; ++dev) body((dev + t) & 3, (r + t) & 1);
        });
    for (auto& t : ts) t.join();
    for (int dev = 0; dev < 4; ++dev)
        for (int k = 0; k < 2; ++k)
            if (runs[dev][k] != 1) return 1;  // once per (device, kernel), whatever the threads
    int tries = 0;
    auto failing = [&] { ++tries; return tries < 2 ? cudaErrorInvalidValue : cudaSuccess; };
    if (reg.run(5, fa, 7, failing) != cudaErrorInvalidValue) return 2;
    if (reg.seen(5, fa, 7)) return 3;       // a failed set-up is not recorded
    if (reg.run(5, fa, 7, failing) != cudaSuccess || tries != 2) return 4;
    if (!reg.seen(5, fa, 7) || reg.seen(6, fa, 7) || reg.seen(5, fa, 8)) return 5;
    return 0;
}

attn_status attn_set_alibi(attn_handle h, const float* slopes) {
    if (!h) return ATTN_ERR_INVALID_ARG;
    if (!slopes) {  // back to no bias
        if (h->d_alibi) cudaFree(h->d_alibi);
        h->d_alibi = nullptr;
        h->tp.alibi = nullptr;
        return ATTN_OK;
    }
    for (int a = 0; a < h->Hq; ++a)
        if (!std::isfinite(slopes[a])) return ATTN_ERR_INVALID_ARG;
    if (h->tp.bias) return ATTN_ERR_UNSUPPORTED;  // ALiBi and a bias matrix are exclusive
    if (!h->d_alibi) {
        cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&h->d_alibi), sizeof(float) * h->Hq);
        if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? ATTN_ERR_OOM : ATTN_ERR_CUDA;
    }
    if (cudaMemcpy(h->d_alibi, slopes, sizeof(float) * h->Hq, cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_ERR_CUDA;
    h->tp.alibi = h->d_alibi;
    return ATTN_OK;
}

attn_status attn_set_bias(attn_handle h, const void* bias, int Bb, int Hb, long ld) {
    if (!h) return ATTN_ERR_INVALID_ARG;
    if (!bias) {  // back to no bias
        h->tp.bias = nullptr;
        h->tp.bias_Bb = h->tp.bias_Hb = 0;
        h->tp.bias_ld = 0;
        return ATTN_OK;
    }
    if (!aligned16(bias) || (Bb != 1 && Bb != h->B) || (Hb != 1 && Hb != h->Hq) || ld < h->S || ld % 8 != 0)
        return ATTN_ERR_INVALID_ARG;
    if (h->dtype == ATTN_F32 || h->tp.alibi) return ATTN_ERR_UNSUPPORTED;
    if (!encode_map_bias(&h->tp.tm_bias, bias, ld, h->S, (long)Bb * Hb)) return ATTN_ERR_CUDA;
    h->tp.bias = static_cast<const uint16_t*>(bias);
    h->tp.bias_Bb = Bb;
    h->tp.bias_Hb = Hb;
    h->tp.bias_ld = ld;
    return ATTN_OK;
}

attn_status attn_backward(attn_handle h, const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                          const void* dO, void* dQ, void* dK, void* dV, void* stream_ptr) {
    if (!h || !Q || !K || !V || !O || !LSE || !dO || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
    const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV};
    for (const void* q : ptrs)
        if (!aligned16(q)) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(LSE) & 3u) return ATTN_ERR_INVALID_ARG;
    if (h->dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    const bool lg = h->kind == ATTN_MASK_LOCAL_GLOBAL;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const int nq = (h->S + ATTN_TILE - 1) / ATTN_TILE;
    const int S_pad = nq * ATTN_TILE;
    attn::BwdParams& p = h->bp;
    cudaError_t e = cudaSuccess;
    if (!h->d_lse2) {
        const size_t n = (size_t)h->B * h->Hq * S_pad;
        std::vector<int> items, dq_items, list;
        if (lg) {  // both kernels walk per-tile lists (the global rows and columns break the band)
            std::vector<int> offsets;
            attn::build_lg_pair_lists(h->S, h->window, h->globals, &list, &offsets);
            attn::build_lg_bwd_items(h->B, h->Hq, h->Hkv, h->S, h->d, offsets, &dq_items, &items);
        } else {
            attn_status st = attn::build_kv_schedule(h->S, h->kind, h->window, &items);
            if (st != ATTN_OK) return st;
            dq_items = attn::order_dq_items(h->sched.items, h->sched.n_main, h->Hq, h->Hkv,
                                            attn::dq_kv_group(h->S, h->d));
        }
        h->n_kv_items = (int)(items.size() / ATTN_WORK_INTS);
        h->n_dq_items = (int)(dq_items.size() / ATTN_WORK_INTS);
        if ((e = cudaMalloc(reinterpret_cast<void**>(&h->d_lse2), n * sizeof(float))) != cudaSuccess ||
            (e = cudaMalloc(reinterpret_cast<void**>(&h->d_dvec), n * sizeof(float))) != cudaSuccess ||
            (e = upload(reinterpret_cast<int**>(&h->d_kvwork), items.data(), items.size())) != cudaSuccess ||
            (e = upload(reinterpret_cast<int**>(&h->d_dqwork), dq_items.data(), dq_items.size())) != cudaSuccess ||
            (lg && (e = upload(&h->d_bwdlist, list.data(), list.size())) != cudaSuccess))
            return e == cudaErrorMemoryAllocation ? ATTN_ERR_OOM : ATTN_ERR_CUDA;
        p.list = h->d_bwdlist;
        p.gbits = lg ? h->d_gbits : nullptr;
        p.S = h->S; p.S_pad = S_pad; p.Hq = h->Hq; p.Hkv = h->Hkv; p.group = h->Hq / h->Hkv;
        p.kind = h->kind; p.window = h->window;
        p.scale = h->scale;
        p.scale_log2 = (float)((double)h->scale * 1.4426950408889634);
        p.nlse2 = h->d_lse2; p.nd = h->d_dvec;
        p.err = h->d_err;
        p.watchdog_ns = h->tp.watchdog_ns;
    }
    // tensor maps (re-encoded when a pointer changes)
    const long BHq = (long)h->B * h->Hq, BHkv = (long)h->B * h->Hkv;
    struct M { CUtensorMap* map; const void* ptr; long heads; } maps[] = {
        {&p.tm_q, Q, BHq}, {&p.tm_k, K, BHkv}, {&p.tm_v, V, BHkv}, {&p.tm_do, dO, BHq},
        {&p.tm_dq, dQ, BHq}, {&p.tm_dk, dK, BHkv}, {&p.tm_dv, dV, BHkv}};
    for (int m = 0; m < 7; ++m) {
        if (maps[m].ptr != h->last_bwd[m]) {
            if (!encode_map(maps[m].map, maps[m].ptr, h->d, h->S, maps[m].heads, kTileRows)) return ATTN_ERR_CUDA;
            h->last_bwd[m] = maps[m].ptr;
        }
    }
    p.alibi = h->tp.alibi;  // the forward's ALiBi slopes (attn_set_alibi), or null
    p.bias = h->tp.bias;    // the forward's bias matrix (attn_set_bias), or null
    p.bias_Bb = h->tp.bias_Bb;
    p.bias_Hb = h->tp.bias_Hb;
    p.bias_ld = h->tp.bias_ld;
    attn::BwdPrepParams pp{};
    pp.o = static_cast<const uint16_t*>(O); pp.dout = static_cast<const uint16_t*>(dO); pp.lse = LSE;
    pp.nlse2 = h->d_lse2; pp.nd = h->d_dvec;
    pp.BHq = (int)BHq; pp.S = h->S; pp.S_pad = S_pad; pp.d = h->d;
    if ((e = attn::launch_bwd_prep(pp, stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    p.work = h->d_dqwork;  // one item per (batch x query head, query tile), grouped by kv head
    if ((e = attn::launch_bwd_dq(p, h->d, h->n_dq_items, stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    p.work = h->d_kvwork;
    p.n_items = h->n_kv_items;
    if ((e = attn::launch_bwd_dkdv(p, h->d, (int)BHkv * h->n_kv_items, stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    if (h->debug) {
        int code = 0;
        return attn_poll_device_error(h, &code);
    }
    return ATTN_OK;
}

attn_status attn_set_fp8_descale(attn_handle h, float descale_q, float descale_k, float descale_v) {
    if (!h) return ATTN_ERR_INVALID_ARG;
    if (h->dtype != ATTN_FP8_E4M3) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(descale_q) || !std::isfinite(descale_k) || !std::isfinite(descale_v) || !(descale_q > 0.f) ||
        !(descale_k > 0.f) || !(descale_v > 0.f))
        return ATTN_ERR_INVALID_ARG;
    h->tp.scale_log2 = (float)((double)h->scale * descale_q * descale_k * 1.4426950408889634);
    h->tp.o_scale = descale_v;
    return ATTN_OK;
}

attn_status attn_set_watchdog(attn_handle h, long long limit_ns, int withhold) {
    if (!h || limit_ns <= 0 || (withhold != 0 && withhold != 1)) return ATTN_ERR_INVALID_ARG;
    h->tp.watchdog_ns = limit_ns;
    h->tp.withhold_v = withhold;
    return ATTN_OK;
}

}  // extern "C"
