// attr.h -- raising a kernel's dynamic shared-memory limit once per device.
#pragma once
#include <cuda_runtime.h>

#include <atomic>

namespace moe {

constexpr int kMaxDevices = 64;

// The dynamic shared-memory limit is an attribute of the function on each device: raise kernel's
// limit to `bytes` on the current device unless `done[device]` records that it already holds at
// least that much. Concurrent callers may both set it (the same value): harmless.
template <typename Kernel>
inline cudaError_t raise_smem_limit(Kernel kernel, int bytes, std::atomic<int> (&done)[kMaxDevices])
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const bool tracked = dev >= 0 && dev < kMaxDevices;
    if (tracked && done[dev].load(std::memory_order_acquire) >= bytes)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && tracked) {
        int cur = done[dev].load(std::memory_order_relaxed);
        while (cur < bytes && !done[dev].compare_exchange_weak(cur, bytes, std::memory_order_release))
            ;
    }
    return e;
}

}  // namespace moe
