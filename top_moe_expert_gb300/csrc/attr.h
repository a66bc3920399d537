// attr.h -- per-device host-side facts and one-time kernel attributes.
//
// A kernel's dynamic-shared-memory limit is an attribute of the device
// context: a process that drives several GPUs needs it set on each one, and
// setting it on every launch would cost a driver call per launch.  The SM
// count is cached per device for the same reason.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <unordered_map>

namespace moe {

// Sets func's maximum dynamic shared memory to `bytes` on the current device
// the first time it is asked for that device; `done` is the caller's bitmask
// of devices already set (devices 64 and up are set on every call).  Only for
// kernels whose launches all use the same size.  Returns false when CUDA
// refuses.
inline bool smem_attr_once(std::atomic<uint64_t> &done, const void *func, int bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit))
        return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    if (bit)
        done.fetch_or(bit, std::memory_order_release);
    return true;
}

// The same for call sites that pick one of several kernels at run time:
// the devices already set are kept per kernel in a small map.  `bytes` is the
// call site's upper bound on the kernel's dynamic shared memory (the limit is
// a cap: launches may use less).  Returns false when CUDA refuses.
inline bool smem_attr(const void *func, int bytes)
{
    static std::mutex mu;
    static std::unordered_map<const void *, uint64_t> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit) {
        std::lock_guard<std::mutex> lock(mu);
        auto it = done.find(func);
        if (it != done.end() && (it->second & bit))
            return true;
    }
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    if (bit) {
        std::lock_guard<std::mutex> lock(mu);
        done[func] |= bit;
    }
    return true;
}

// Number of SMs of the current device (cached per device; 148 if CUDA does
// not answer).
inline int device_sm_count()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64) {
        const int n = cache[dev].load(std::memory_order_relaxed);
        if (n > 0)
            return n;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev >= 0 && dev < 64)
        cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace moe
