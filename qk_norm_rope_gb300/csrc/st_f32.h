// Parameter block and launchers of the exact-fp32 kernels (st_f32.cu).
#pragma once
#include <cuda_runtime.h>
#include "st_common.cuh"

namespace st {

constexpr int kF32Tile = 64;  // rows of the fp32 path's query and key tiles

struct F32Params {
  Common c;  // q, k, v (all fp32), norm weights, rotary tables, mask, scale, sizes
  // forward outputs
  float* o;  // [B, Sq, H, D]
  int64_t o_sb, o_ss, o_sh;
  float* lse;  // [B, H, Sq]
  // backward inputs and outputs
  const float* lse_in;  // [B, H, Sq], from the forward
  const float* delta;   // [B, H, Sq], rowsum(dO * O) from the pre kernel
  const float* dout;    // [B, Sq, H, D]
  int64_t do_sb, do_ss, do_sh;
  float* dq;
  int64_t dq_sb, dq_ss, dq_sh;
  float* dk;  // [B, Skv, Hkv, D]
  int64_t dk_sb, dk_ss, dk_sh;
  float* dv;
  int64_t dv_sb, dv_ss, dv_sh;
  float* dwq_part;  // [B, H, ceil(Sq / 64), D]
  float* dwk_part;  // [B, Hkv, ceil(Skv / 64), D]
};

// Forward: O and the log-sum-exp.
cudaError_t launch_f32_fwd(const F32Params& p, cudaStream_t stream);
// Backward, with Delta in place (the pre kernel): dk, dv and the k weight
// partials (a kernel over key tiles, S_kv > 0); dq and the q weight partials
// (a kernel over query tiles, S_q > 0).
cudaError_t launch_f32_bwd_kv(const F32Params& p, cudaStream_t stream);
cudaError_t launch_f32_bwd_q(const F32Params& p, cudaStream_t stream);

}  // namespace st
