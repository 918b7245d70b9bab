// attn_forward_noalloc: the bf16 forward pass without any device allocation.
//
// Some callers cannot call cudaMalloc: code that runs inside a memory pool it
// does not own, runtimes that forbid allocation once a model is loaded, or
// processes that must keep their device footprint fixed after start-up.  For
// them this entry point takes the problem description and the caller's Q, K,
// V, O, LSE buffers and keeps every other device byte it needs (error word,
// work list, global-token list, bits and per-tile split, partial results and
// arrival counters of the global-row chunks) in one file-scope __device__ array of
// ATTN_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds
// until the process exits.
//
// The first call on a device looks up the array's device address with
// cudaGetSymbolAddress (once per device, with that device current); make that
// first call before any stream capture.  All calls share the array and it
// keeps the last call's contents, so calls that overlap on the GPU (on two
// streams, or on two host threads) race and must be serialised by the caller.
// The schedule reaches the device inside kernel parameters (a small copy
// kernel per 30 KiB), which the launch itself copies: no host buffer is read
// after the call returns.  The error word collects the watchdog bits of every
// call until attn_forward_noalloc_poll_error reads and clears it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
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

// Byte offset of the error word inside the scratch array (it stays at the front for every problem).
constexpr size_t kOffErr = 0;

// Watchdog settings of this entry point (attn_forward_noalloc_set_watchdog).
std::atomic<long long> g_watchdog_ns{2000000000LL};
std::atomic<int> g_withhold_v{0};

// Host words passed by value: kernel parameters are copied when the launch is made.
constexpr int kUploadWords = 7680;  // 30 KiB of payload (kernel parameters hold up to 32,764 bytes)
struct UploadChunk {
    unsigned* dst;
    int n;
    unsigned w[kUploadWords];
};

__global__ void __launch_bounds__(256) noalloc_upload_kernel(const __grid_constant__ UploadChunk c) {
    for (int k = threadIdx.x; k < c.n; k += blockDim.x) c.dst[k] = c.w[k];
}

// Copies n words from the host to dst on `stream`, in launches of kUploadWords words.
cudaError_t upload_words(unsigned* dst, const void* src, size_t n, cudaStream_t stream) {
    UploadChunk c;
    const unsigned* s = static_cast<const unsigned*>(src);
    for (size_t k = 0; k < n; k += kUploadWords) {
        c.dst = dst + k;
        c.n = (int)std::min<size_t>(kUploadWords, n - k);
        std::memcpy(c.w, s + k, (size_t)c.n * sizeof(unsigned));
        noalloc_upload_kernel<<<1, 256, 0, stream>>>(c);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

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
    // per query tile: the globals before its band of key tiles, and before the band's end
    std::vector<int> gsplit((size_t)nk * 2, 0);
    for (int t = 0; t < n_first; ++t) {
        const int* it = &items[(size_t)t * ATTN_WORK_INTS];
        const long lo = std::min<long>((long)it[2] * ATTN_TILE, S), hi = std::min<long>((long)it[3] * ATTN_TILE, S);
        gsplit[(size_t)it[1] * 2] = (int)(std::lower_bound(G.begin(), G.end(), lo) - G.begin());
        gsplit[(size_t)it[1] * 2 + 1] = (int)(std::lower_bound(G.begin(), G.end(), hi) - G.begin());
    }

    // carve the fixed scratch area; refuse problems that do not fit
    const size_t off_work = 256;
    const size_t off_glob = off_work + round256(items.size() * sizeof(int));
    const size_t off_bits = off_glob + round256((size_t)nG * sizeof(int));
    // key chunks of the global rows: the chunk index is int [7] of those items
    int n_chunks = 1;
    for (int t = n_first; t < n_items; ++t) n_chunks = std::max(n_chunks, items[(size_t)t * ATTN_WORK_INTS + 7] + 1);
    const int n_gtiles = (nG + ATTN_TILE - 1) / ATTN_TILE;
    const size_t part_rows = n_chunks > 1 ? (size_t)B * Hq * nG * n_chunks : 0;
    const size_t n_ctr = n_chunks > 1 ? (size_t)B * Hq * n_gtiles : 0;
    const size_t off_gsplit = off_bits + round256(bits.size() * sizeof(unsigned));
    const size_t off_part_o = off_gsplit + round256(gsplit.size() * sizeof(int));
    const size_t off_part_lse = off_part_o + round256(part_rows * d_k * sizeof(float));
    const size_t off_ctr = off_part_lse + round256(part_rows * sizeof(float));
    const size_t total = off_ctr + round256(n_ctr * sizeof(unsigned));
    if (total > kScratchBytes) return ATTN_ERR_UNSUPPORTED;

    void* base = nullptr;
    if ((st = scratch_address(&base)) != ATTN_OK) return st;
    unsigned char* sc = static_cast<unsigned char*>(base);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    // the schedule, in kernel parameters; the arrival counters must start at zero
    if (upload_words(reinterpret_cast<unsigned*>(sc + off_work), items.data(), items.size(), stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (nG > 0 && upload_words(reinterpret_cast<unsigned*>(sc + off_glob), G.data(), G.size(), stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (upload_words(reinterpret_cast<unsigned*>(sc + off_bits), bits.data(), bits.size(), stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (upload_words(reinterpret_cast<unsigned*>(sc + off_gsplit), gsplit.data(), gsplit.size(), stream) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    if (n_ctr > 0 && cudaMemsetAsync(sc + off_ctr, 0, n_ctr * sizeof(unsigned), stream) != cudaSuccess)
        return ATTN_ERR_CUDA;

    attn::TcParams p{};
    constexpr unsigned T = ATTN_TILE;
    const unsigned kvb = attn::tc_kv_box_rows(d_k);
    if (!map3d(&p.tm_q, Q, d_k, S, (long)B * Hq, T) || !map3d(&p.tm_k, K, d_k, S, (long)B * Hkv, kvb) ||
        !map3d(&p.tm_v, V, d_k, S, (long)B * Hkv, kvb) || !map3d(&p.tm_o, O, d_k, S, (long)B * Hq, T))
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
    p.gsplit = reinterpret_cast<const int2*>(sc + off_gsplit);
    p.q = static_cast<const uint16_t*>(Q);
    p.k = static_cast<const uint16_t*>(K);
    p.v = static_cast<const uint16_t*>(V);
    p.o = O;
    p.lse = LSE;
    p.err = reinterpret_cast<int*>(sc + kOffErr);
    p.watchdog_ns = g_watchdog_ns.load();
    p.withhold_v = g_withhold_v.load();
    p.n_chunks = n_chunks;
    p.part_o = n_chunks > 1 ? reinterpret_cast<float*>(sc + off_part_o) : nullptr;
    p.part_lse = n_chunks > 1 ? reinterpret_cast<float*>(sc + off_part_lse) : nullptr;
    p.counters = n_chunks > 1 ? reinterpret_cast<unsigned*>(sc + off_ctr) : nullptr;
    p.n_gtiles = n_gtiles;
    p.fp8 = 0;        // bf16 inputs
    p.o_scale = 1.f;  // no output factor
    p.alibi = nullptr;
    p.bias = nullptr;

    p.item_offset = 0;
    if (attn::launch_tc_forward(p, d_k, n_items, stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

extern "C" attn_status attn_forward_noalloc_poll_error(int* code) {
    if (!code) return ATTN_ERR_INVALID_ARG;
    *code = 0;
    void* base = nullptr;
    const attn_status st = scratch_address(&base);
    if (st != ATTN_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned char* sc = static_cast<unsigned char*>(base);
    if (cudaMemcpy(code, sc + kOffErr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (*code != 0 && cudaMemset(sc + kOffErr, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    return *code ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
}

extern "C" attn_status attn_forward_noalloc_set_watchdog(long long limit_ns, int withhold) {
    if (limit_ns <= 0 || (withhold != 0 && withhold != 1)) return ATTN_ERR_INVALID_ARG;
    g_watchdog_ns.store(limit_ns);
    g_withhold_v.store(withhold);
    return ATTN_OK;
}
