// Backward of the scan from a starting state with document resets
// (mamba_selective_scan_bwd_ex): a.f.h0 and a.f.reset as for the forward;
// dh0 [batch, dim, N] (or nullptr) receives the gradient of h0.
#pragma once

#include "common.cuh"

namespace mamba {

cudaError_t launch_scan_bwd_ex(const ScanBwdArgs& a, float* dh0, bool bf16, cudaStream_t stream);

}  // namespace mamba
