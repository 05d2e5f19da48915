// Launchers of the kernels that live in their own translation units.
#pragma once
#include <cuda_runtime.h>
#include "st_common.cuh"

namespace st {
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t stream);
}  // namespace st
