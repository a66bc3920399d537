// attr.h -- per-device, one-time kernel attribute setting (host code).
//
// A kernel's dynamic-shared-memory limit is an attribute of the device
// context: a process that drives several GPUs needs it set on each one, and
// setting it on every launch would cost a driver call per launch.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace moe {

// Sets func's maximum dynamic shared memory to `bytes` on the current device
// the first time it is asked for that device; `done` is the caller's bitmask
// of devices already set (devices 64 and up are set on every call).  Returns
// false when CUDA refuses.
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

}  // namespace moe
