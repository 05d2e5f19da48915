// Parameter blocks and launchers of the auxiliary kernels.
#pragma once
#include <algorithm>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include "st_common.cuh"

namespace st {

// Control words at the start of the workspace, zeroed by the table kernel
// (always the first launch of a call).
enum { kCtrlAnyFalse = 0, kCtrlClassifyDone = 1, kCtrlDwDone = 2 /* +0 q, +1 k */, kCtrlWords = 8 };
constexpr int kDwChunk = 32;  // weight-gradient partials summed per block
constexpr int kPostBlockRows = 64;   // rows of one dq_post block (and of one dW_q partial)

inline int dw_reduce_blocks(int n_q, int n_k) {
  const int a = (n_q + kDwChunk - 1) / kDwChunk, b = (n_k + kDwChunk - 1) / kDwChunk;
  return std::max(1, std::max(a, b));
}

// st_dtype codes of a caller table (the C header's ST_BF16, ST_F16, ST_F32).
constexpr int kTabBF16 = 0, kTabF16 = 1, kTabF32 = 2;

struct TableParams {
  const void* ids;
  int ids_f32;
  int64_t i_sb, i_ss, i_sa;  // element strides of ids [Bt, S, A]
  // table form (cos non-null): the caller's pair-duplicated cos/sin [Bt, S, D]
  const void* cos;
  const void* sin;
  int tab_dtype;             // st_dtype of cos and sin (fp32, bf16 or fp16)
  int64_t c_sb, c_ss, c_sd;  // element strides of cos (0 on a broadcast batch)
  int64_t s_sb, s_ss, s_sd;  // element strides of sin
  int Bt, S;
  double omega[kPairs];      // frequency of each pair
  int axis_of[kPairs];       // axis that owns each pair
  float2* out;               // [Bt, S, 64] (cos, sin) fp32
  __half2* out16;            // [Bt, S, 64] (cos, sin) fp16, read by the operand prologues
  unsigned* ctrl;            // zeroed when non-null
  unsigned* zero;            // n_zero further words zeroed (the forward's K' publication flags), or null
  int64_t n_zero;
};

struct ClassifyParams {
  const uint8_t* mask;
  int64_t m_sb, m_sh, m_sq;  // element strides, 0 on broadcast dims
  int Bm, Hm, Sqm, Skv, nQtm, nKt;
  uint8_t* flags;            // [Bm, Hm, nQtm, nKt]
  unsigned* ctrl;
  unsigned long long* counters;
};

struct PreParams {
  const void* o;
  int64_t o_sb, o_ss, o_sh;
  int o_dt;       // element type of O and dO (kDtBF16, kDtF16 or kDtF32)
  const void* dout;
  int64_t do_sb, do_ss, do_sh;
  float* delta;   // [B, H, Sq]
  float* dq_acc;  // [B, Sq, H, D], zeroed (nullptr: none to zero)
  unsigned* ctrl; // control words: the weight-gradient counters are cleared
  int B, H, Sq;
};

struct PostParams {
  const float* dq_acc;
  RowTensor q;
  const float2* tab_q;
  int64_t tab_q_sb;
  const float* wq;
  float eps;
  void* dq;
  int64_t dq_sb, dq_ss, dq_sh;
  int dq_dt;
  float* dwq_part;  // [n_blocks, D]
  int B, H, Sq;
};

// Q' rows for a backward that does not reuse a forward's workspace: the
// forward kernel's q prologue (RMSNorm with the q weights, rotation, rounding
// to the 16-bit operand type) as a row kernel into [B, Sq, H, D].
struct QPrimeParams {
  RowTensor q;
  const float2* tab;      // fp32 (cos, sin) rows: fp32 q, as the forward's fp32 prologue
  const __half2* tab16;   // fp16 (cos, sin) rows: 16-bit q, as the forward's TMA-staged prologue
  int64_t tab_sb;         // pairs between the tables of two samples (0: shared)
  const float* w;
  float eps;
  void* out;              // [B, Sq, H, D] contiguous, 16-bit operand type
  int f16;                // operand type: 1 fp16, 0 bf16
  int B, H, Sq;
};

struct DwParams {
  const float* dwq_part;
  const float* dwk_part;
  int n_q, n_k;
  float* scratch;  // [2, blocks, D]
  unsigned* ctrl;
  float* dwq;
  float* dwk;
};

cudaError_t launch_table(const TableParams& p, cudaStream_t stream);
cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t stream);
cudaError_t launch_bwd_pre(const PreParams& p, cudaStream_t stream);
cudaError_t launch_dq_post(const PostParams& p, cudaStream_t stream);
cudaError_t launch_dw_reduce(const DwParams& p, cudaStream_t stream);
cudaError_t launch_qprime(const QPrimeParams& p, cudaStream_t stream);
cudaError_t launch_wait_probe(unsigned* status, unsigned long long* counters, long long budget, cudaStream_t stream);

}  // namespace st
