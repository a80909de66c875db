// Programmatic dependent launch (sm_90 and later).
//
// A kernel launched with the programmatic-serialization attribute may start
// while the kernel before it on the stream drains: its CTAs take the slots
// that the earlier grid's CTAs free.  Such a kernel calls
// grid_dependency_wait() before its first global memory access: it returns
// once the earlier grid has completed and its memory operations are visible,
// so the ordering the stream promises holds for every byte the kernel reads
// or writes.  grid_launch_dependents() lets the next such launch be scheduled
// as this grid's CTAs exit.  Without the attribute both are no-ops.
#pragma once

#include <atomic>
#include <cstdlib>
#include <utility>

#include <cuda_runtime.h>

namespace mamba {

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` with the programmatic-serialization attribute unless the
// environment variable `off_var` is set to "0".
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, const char* off_var, Args&&... args) {
    const char* v = off_var ? getenv(off_var) : nullptr;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = (v && v[0] == '0') ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Per-device cache of a kernel's launch shape: the SM count and the resident
// CTAs per SM (whose query, with the shared-memory attribute it needs, costs
// more host time than a short kernel's launch).  One cache per call site;
// devices beyond kMaxCachedDevices are queried on every call.
constexpr int kMaxCachedDevices = 64;
struct LaunchShapeCache {
    std::atomic<long long> v[kMaxCachedDevices];  // (sms << 32) | per_sm; 0 = not known yet
};

// query(int* sms, int* per_sm) -> bool fills both on success.
template <typename Query>
bool cached_launch_shape(LaunchShapeCache& cache, Query&& query, int* sms, int* per_sm) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (dev < 0 || dev >= kMaxCachedDevices) return query(sms, per_sm);
    long long x = cache.v[dev].load(std::memory_order_acquire);
    if (x == 0) {
        if (!query(sms, per_sm) || *sms <= 0 || *per_sm <= 0) return false;
        x = (static_cast<long long>(*sms) << 32) | static_cast<unsigned>(*per_sm);
        cache.v[dev].store(x, std::memory_order_release);
    }
    *sms = static_cast<int>(x >> 32);
    *per_sm = static_cast<int>(x & 0xffffffffLL);
    return true;
}

}  // namespace mamba
