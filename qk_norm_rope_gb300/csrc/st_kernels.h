// Launchers of the kernels that live in their own translation units.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>
#include "st_common.cuh"

namespace st {

// The attention kernels of each 16-bit operand type are compiled in their own
// translation unit (st_fwd.cu / st_bwd.cu: bf16; st_fwd_f16.cu / st_bwd_f16.cu:
// fp16).
cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_f16(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_f16(const BwdParams& p, cudaStream_t stream);

inline cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  return p.c.f16 ? launch_fwd_f16(p, stream) : launch_fwd_bf16(p, stream);
}
inline cudaError_t launch_bwd(const BwdParams& p, cudaStream_t stream) {
  return p.c.f16 ? launch_bwd_f16(p, stream) : launch_bwd_bf16(p, stream);
}

// Raises the kernel's dynamic shared-memory limit to `bytes`, once per device
// (a bit per device in `done`, set with an atomic or; two threads racing on
// the first launch both set the same attribute, which is harmless).
template <class Kernel>
cudaError_t opt_in_smem(Kernel kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  done.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

}  // namespace st
