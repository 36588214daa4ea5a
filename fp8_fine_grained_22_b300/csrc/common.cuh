// common.cuh -- host-side helpers shared by the fp8fg translation units:
// status mapping, alignment checks and the per-device SM-count cache.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fp8fg.h"

namespace fp8fg {

inline bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Status of the launch just made on this thread.
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

// Number of SMs of the current device (cached per device), or -1.
inline int sm_count_current(int* dev_out = nullptr) {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    if (dev_out) *dev_out = dev;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            return -1;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace fp8fg
