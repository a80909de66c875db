// Library-owned stream-ordered memory pools (see scratch_pool.cuh).
#include "scratch_pool.cuh"

#include <cstdint>
#include <cstdlib>
#include <mutex>

namespace mamba {
namespace {

constexpr int kMaxPoolDevices = 64;

uint64_t retain_bytes() {
    const char* v = getenv("MAMBA_SCRATCH_RETAIN_MB");
    if (!v || !*v) return UINT64_MAX;
    const long long mb = atoll(v);
    return mb <= 0 ? 0 : static_cast<uint64_t>(mb) << 20;
}

// The pool of device `dev`, created on first use; nullptr if that failed.
cudaMemPool_t pool_for(int dev) {
    static std::mutex mu;
    static cudaMemPool_t pools[kMaxPoolDevices] = {};
    static bool tried[kMaxPoolDevices] = {};
    if (dev < 0 || dev >= kMaxPoolDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!tried[dev]) {
        tried[dev] = true;
        const bool pending = cudaPeekAtLastError() != cudaSuccess;
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) == cudaSuccess) {
            uint64_t keep = retain_bytes();
            if (cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep) ==
                cudaSuccess) {
                pools[dev] = p;
            } else {
                cudaMemPoolDestroy(p);
            }
        }
        // a failed creation leaves the default pool in use; it clears the
        // error it set, but only when none was pending before it
        if (!pools[dev] && !pending) cudaGetLastError();
    }
    return pools[dev];
}

}  // namespace

cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    cudaMemPool_t pool = pool_for(dev);
    return pool ? cudaMallocFromPoolAsync(ptr, bytes, pool, stream)
                : cudaMallocAsync(ptr, bytes, stream);
}

cudaError_t scratch_free(void* ptr, cudaStream_t stream) { return cudaFreeAsync(ptr, stream); }

}  // namespace mamba
