// Per-device, thread-safe "first time" registry for host-side kernel set-up.
//
// Kernel attributes such as the dynamic shared-memory opt-in belong to the device
// context: setting one while device 0 is current does nothing for device 1.  A
// process-wide flag per kernel would skip the set-up on the second GPU of a process
// (and two host threads racing on a plain bool is a data race), so every launcher asks
// this registry instead, keyed by (device, kernel, value).
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <tuple>

namespace attn {

class DeviceOnce {
public:
    // Runs fn() unless it already succeeded for (device, key, value); returns its result.
    // Holds the lock while fn runs, so two threads never set up the same entry at once.
    template <class F>
    cudaError_t run(int device, const void* key, long value, F&& fn) {
        std::lock_guard<std::mutex> lock(mu_);
        const auto k = std::make_tuple(device, key, value);
        if (done_.count(k)) return cudaSuccess;
        const cudaError_t e = fn();
        if (e == cudaSuccess) done_.insert(k);
        return e;
    }
    bool seen(int device, const void* key, long value) {
        std::lock_guard<std::mutex> lock(mu_);
        return done_.count(std::make_tuple(device, key, value)) != 0;
    }

private:
    std::mutex mu_;
    std::set<std::tuple<int, const void*, long>> done_;
};

// The process-wide registry (one instance shared by every translation unit).
DeviceOnce& device_once();

// Opts `func` in to `bytes` of dynamic shared memory on the current device, once per device.
inline cudaError_t smem_opt_in(const void* func, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return device_once().run(dev, func, bytes, [&] {
        return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    });
}

// Streaming multiprocessors of the current device (0 if it cannot be queried).
inline int current_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace attn
