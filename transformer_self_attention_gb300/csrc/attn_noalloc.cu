// attn_forward_noalloc: the bf16 forward pass without any device allocation.
//
// Some callers cannot call cudaMalloc: code that runs inside a memory pool it
// does not own, runtimes that forbid allocation once a model is loaded, or
// processes that must keep their device footprint fixed after start-up.  For
// them this entry point takes the problem description and the caller's Q, K,
// V, O, LSE buffers and keeps every other device byte it needs (error word,
// work list, global-token list and bits, gathered global rows) in one
// file-scope __device__ array of ATTN_NOALLOC_SCRATCH_BYTES, which every GPU
// that loads the library holds until the process exits.
//
// The first call on a device looks up the array's device address with
// cudaGetSymbolAddress (once per device, with that device current); make that
// first call before any stream capture.  All calls share the array and it
// keeps the last call's contents, so calls that overlap on the GPU (on two
// streams, or on two host threads) race and must be serialised by the caller.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "attn.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_addr_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
attn_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_addr_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return ATTN_OK;
}

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

// bf16 [heads, rows, d] map, box {64, box_rows, 1}, 128-byte swizzle (the layout the kernel expects)
bool map3d(CUtensorMap* m, const void* base, int d, long rows, long heads, unsigned box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" attn_status attn_forward_noalloc(int B, int Hq, int Hkv, int S, int d_k, float scale,
                                            attn_mask_kind kind, int window, const int* global_idx, int n_global,
                                            const void* Q, const void* K, const void* V, void* O, float* LSE,
                                            void* stream_ptr) {
    if (!Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                          reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O);
    if ((mis & 15u) || (reinterpret_cast<uintptr_t>(LSE) & 3u)) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;

    // the host schedule (validates the shape and mask arguments)
    int n_items = 0, n_first = 0;
    attn_status st = attn_schedule_host(B, Hq, Hkv, S, kind, window, global_idx, n_global, nullptr, 0, &n_items,
                                        &n_first);
    if (st != ATTN_OK) return st;
    if (d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED;
    std::vector<int> items((size_t)n_items * ATTN_WORK_INTS);
    st = attn_schedule_host(B, Hq, Hkv, S, kind, window, global_idx, n_global, items.data(), n_items, &n_items,
                            &n_first);
    if (st != ATTN_OK) return st;
    std::vector<int> G(global_idx, global_idx + n_global);
    std::sort(G.begin(), G.end());
    G.erase(std::unique(G.begin(), G.end()), G.end());
    const int nG = (int)G.size();
    const int nk = (S + ATTN_TILE - 1) / ATTN_TILE;
    std::vector<unsigned> bits((size_t)nk * 4, 0u);
    for (int g : G) bits[(size_t)(g / ATTN_TILE) * 4 + (g % ATTN_TILE) / 32] |= 1u << (g % 32);

    // carve the fixed scratch area; refuse problems that do not fit
    const size_t off_err = 0;
    const size_t off_work = 256;
    const size_t off_glob = off_work + round256(items.size() * sizeof(int));
    const size_t off_bits = off_glob + round256((size_t)nG * sizeof(int));
    const size_t off_qg = off_bits + round256(bits.size() * sizeof(unsigned));
    const size_t qg_bytes = (size_t)B * Hq * nG * d_k * 2, kg_bytes = (size_t)B * Hkv * nG * d_k * 2;
    const size_t off_kg = off_qg + round256(qg_bytes);
    const size_t off_vg = off_kg + round256(kg_bytes);
    // key chunks of the global-row pass: the chunk index is int [7] of those items
    int n_chunks = 1;
    for (int t = n_first; t < n_items; ++t) n_chunks = std::max(n_chunks, items[(size_t)t * ATTN_WORK_INTS + 7] + 1);
    const size_t part_rows = n_chunks > 1 ? (size_t)B * Hq * nG * n_chunks : 0;
    const size_t off_part_o = off_vg + round256(kg_bytes);
    const size_t off_part_lse = off_part_o + round256(part_rows * d_k * sizeof(float));
    const size_t total = off_part_lse + round256(part_rows * sizeof(float));
    if (total > kScratchBytes) return ATTN_ERR_UNSUPPORTED;

    void* base = nullptr;
    if ((st = scratch_address(&base)) != ATTN_OK) return st;
    unsigned char* sc = static_cast<unsigned char*>(base);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    // the error word must start at zero; everything else is fully overwritten below
    if (cudaMemsetAsync(sc + off_err, 0, sizeof(int), stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemcpyAsync(sc + off_work, items.data(), items.size() * sizeof(int), cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    if (nG > 0 && cudaMemcpyAsync(sc + off_glob, G.data(), (size_t)nG * sizeof(int), cudaMemcpyHostToDevice,
                                  stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (cudaMemcpyAsync(sc + off_bits, bits.data(), bits.size() * sizeof(unsigned), cudaMemcpyHostToDevice,
                        stream) != cudaSuccess)
        return ATTN_ERR_CUDA;

    attn::TcParams p{};
    constexpr unsigned T = ATTN_TILE;
    if (!map3d(&p.tm_q, Q, d_k, S, (long)B * Hq, T) || !map3d(&p.tm_k, K, d_k, S, (long)B * Hkv, T) ||
        !map3d(&p.tm_v, V, d_k, S, (long)B * Hkv, T) || !map3d(&p.tm_o, O, d_k, S, (long)B * Hq, T))
        return ATTN_ERR_CUDA;
    if (nG > 0 && (!map3d(&p.tm_qg, sc + off_qg, d_k, nG, (long)B * Hq, T) ||
                   !map3d(&p.tm_kg, sc + off_kg, d_k, nG, (long)B * Hkv, T) ||
                   !map3d(&p.tm_vg, sc + off_vg, d_k, nG, (long)B * Hkv, T)))
        return ATTN_ERR_CUDA;
    p.work = reinterpret_cast<const int4*>(sc + off_work);
    p.S = S; p.Hq = Hq; p.Hkv = Hkv; p.group = Hq / Hkv;
    p.kind = kind;
    p.window = (kind == ATTN_MASK_SLIDING || kind == ATTN_MASK_CAUSAL_SLIDING || kind == ATTN_MASK_LOCAL_GLOBAL)
                   ? window : 0;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.globals = reinterpret_cast<const int*>(sc + off_glob);
    p.n_global = nG;
    p.global_bits = reinterpret_cast<const unsigned*>(sc + off_bits);
    p.o = O;
    p.lse = LSE;
    p.err = reinterpret_cast<int*>(sc + off_err);
    p.watchdog_ns = 2000000000LL;
    p.withhold_v = 0;
    p.n_chunks = n_chunks;
    p.part_o = n_chunks > 1 ? reinterpret_cast<float*>(sc + off_part_o) : nullptr;
    p.part_lse = n_chunks > 1 ? reinterpret_cast<float*>(sc + off_part_lse) : nullptr;

    if (nG > 0) {
        attn::GatherParams g{};
        g.q = static_cast<const uint16_t*>(Q); g.k = static_cast<const uint16_t*>(K);
        g.v = static_cast<const uint16_t*>(V);
        g.qg = reinterpret_cast<uint16_t*>(sc + off_qg); g.kg = reinterpret_cast<uint16_t*>(sc + off_kg);
        g.vg = reinterpret_cast<uint16_t*>(sc + off_vg);
        g.globals = p.globals; g.n_global = nG;
        g.BHq = B * Hq; g.BHkv = B * Hkv; g.S = S; g.d = d_k;
        if (attn::launch_gather_globals(g, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    }
    p.item_offset = 0;
    if (attn::launch_tc_forward(p, d_k, n_first, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    if (n_items > n_first) {
        p.item_offset = n_first;
        if (attn::launch_tc_forward(p, d_k, n_items - n_first, stream) != cudaSuccess) return ATTN_ERR_CUDA;
        if (n_chunks > 1) {
            attn::MergeParams mp{};
            mp.part_o = p.part_o; mp.part_lse = p.part_lse;
            mp.o = static_cast<uint16_t*>(O); mp.lse = LSE;
            mp.globals = p.globals; mp.n_global = nG; mp.n_chunks = n_chunks;
            mp.BHq = B * Hq; mp.S = S; mp.d = d_k;
            if (attn::launch_merge_global_rows(mp, stream) != cudaSuccess) return ATTN_ERR_CUDA;
        }
    }
    return ATTN_OK;
}
