// Stream-ordered scratch memory for the kernels' temporary buffers (the
// carried states of a time-split scan, the backward's checkpoints).
//
// Allocations come from a memory pool the library creates on each device.
// The device's default pool returns freed memory to the driver at every
// synchronisation point, and the next call then pays for mapping it again
// (about 2 ms for the backward's 268 MB of checkpoints); this pool keeps what
// it holds mapped across synchronisations, up to MAMBA_SCRATCH_RETAIN_MB
// megabytes (all of it when the variable is unset).  If the pool cannot be
// created the device's default pool is used.
#pragma once

#include <cstddef>

#include <cuda_runtime.h>

namespace mamba {

// Like cudaMallocAsync / cudaFreeAsync on `stream`.
cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t stream);
cudaError_t scratch_free(void* ptr, cudaStream_t stream);

}  // namespace mamba
