// common.cuh -- host-side helpers shared by the fp8fg translation units:
// status mapping, alignment checks, the per-device SM-count cache and the
// per-context cache of values that belong to a CUDA context (kernel
// attributes, device addresses of the library's own __device__ arrays).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/fp8fg.h"

namespace fp8fg {

inline bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// The C ABI's status type from the int statuses used internally.
inline fp8_status to_status(int v) { return static_cast<fp8_status>(v); }

// Status of the launch just made on this thread.
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

// Number of SMs of the current device (cached per device; a device's SM
// count never changes), or -1.  Safe under concurrent first calls: every
// thread that finds the slot empty stores the same value.
inline int sm_count_current(int* dev_out = nullptr) {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return -1;
    }
    if (dev_out) *dev_out = dev;
    int n = cache[dev].load(std::memory_order_acquire);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0) {
            (void)cudaGetLastError();
            return -1;
        }
        cache[dev].store(n, std::memory_order_release);
    }
    return n;
}

// Unique id of the CUDA context current on this thread (the driver's
// cuCtxGetId, looked up once through the runtime, so that the library needs
// no link-time dependency on libcuda).  Returns false when no context is
// current yet or the id cannot be read.  Ids are never reused within a
// process: a context re-created after cudaDeviceReset, or a context the
// caller created with the driver API, gets a new one.
inline bool current_context_id(unsigned long long* id) {
    struct Fns {
        PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
        PFN_cuCtxGetId_v12000 get_id = nullptr;
    };
    static const Fns fns = [] {
        Fns f;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        (void)cudaGetLastError();
        return f;
    }();
    if (fns.get_current == nullptr || fns.get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return fns.get_id(ctx, id) == CUDA_SUCCESS;
}

// A value that belongs to the CUDA context current on the calling thread,
// computed on first use in each context and cached per device ordinal
// together with the id of the context it was computed in.  A call in another
// context of the same device (a driver-API context, or the primary context
// re-created after cudaDeviceReset) recomputes it.  All access is under a
// mutex, so concurrent first calls from several host threads are safe.
template <typename T>
class ContextCache {
  public:
    // Returns FP8_OK and *out, computing it with make(T*) -> int status when
    // this (device, context) has no cached value yet.  make runs with the
    // context current; a failed make caches nothing.
    template <typename Make>
    int get(T* out, Make make) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
            (void)cudaGetLastError();
            return FP8_ERR_CUDA;
        }
        unsigned long long id = 0;
        const bool have_id = current_context_id(&id);
        std::lock_guard<std::mutex> lock(mu_);
        Slot& s = slots_[dev];
        if (have_id && s.valid && s.ctx == id) {
            *out = s.value;
            return FP8_OK;
        }
        T v{};
        const int st = make(&v);
        if (st != FP8_OK) {
            (void)cudaGetLastError();  // leave no sticky error for the next call
            return st;
        }
        // make() may have created the primary context: read the id again
        unsigned long long id2 = 0;
        if (current_context_id(&id2)) {
            s.ctx = id2;
            s.value = v;
            s.valid = true;
        }
        *out = v;
        return FP8_OK;
    }

  private:
    struct Slot {
        unsigned long long ctx = 0;
        T value{};
        bool valid = false;
    };
    std::mutex mu_;
    Slot slots_[kMaxDevices];
};

// Device address of the library's error word (the one fp8_device_error reads
// and clears) in the current context; nullptr if it cannot be looked up.
unsigned* device_error_word();

}  // namespace fp8fg
