// launch_util.h -- host helpers shared by the launchers.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace rmsn {

// Lets `func` use up to the device's opt-in maximum of dynamic shared memory.
// Done once per kernel and device (one bit per device in `mask`).
inline cudaError_t allow_max_dynamic_smem(const void *func, std::atomic<uint64_t> &mask) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    mask.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

}  // namespace rmsn
