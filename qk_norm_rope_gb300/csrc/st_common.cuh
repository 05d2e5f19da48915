// Device-side parameter blocks and row helpers shared by the kernels.
#pragma once
#include <cstdint>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include "st_ptx.cuh"

namespace st {

constexpr int kD = 128;        // head dimension handled by the kernels
constexpr int kTile = 128;     // rows of a query tile and of a key tile
constexpr int kPairs = kD / 2; // rotation pairs per row
constexpr uint32_t kTileBytes = kTile * kD * 2;  // one bf16 operand tile (two 128B-swizzled halves)
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 64-column half: 128 rows x 128 B

// Tile classes of a bool mask, one byte per (b|1, h|1, q-tile|1, k-tile).
enum : uint8_t { kTileMixed = 0, kTileAllTrue = 1, kTileAllFalse = 2 };
enum MaskKind : int { kMaskNone = 0, kMaskBool = 1, kMaskF32 = 2, kMaskBF16 = 3 };

// Device status word bits.
enum : unsigned { kStatusTimeout = 1u, kStatusLayout = 2u };

// Device-side counters (indices into a uint64 array).
enum { kCtrMaskAllTrue = 0, kCtrTilesSkipped = 1, kCtrTilesTotal = 2, kCtrTimeouts = 3, kNumCounters = 8 };

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Element types of rows in global memory (the codes of st_dtype).
enum : int { kDtBF16 = 0, kDtF16 = 1, kDtF32 = 2 };

struct RowTensor {  // [B, S, H, D] view with unit stride on D
  const void* p;
  int64_t sb, ss, sh;
  int dt;  // kDtBF16, kDtF16 or kDtF32
};

struct Common {
  RowTensor q, k, v;
  const float* wq;
  const float* wk;
  float eps;
  const float2* tab_q;  // [Bt_q, Sq, 64] (cos, sin)
  const float2* tab_k;  // [Bt_k, Skv, 64]
  int64_t tab_q_sb, tab_k_sb;  // batch stride in float2 (0 when shared by the batch)
  const __half2* tab16_q;      // the same tables in fp16 (same strides), for the prologues
  const __half2* tab16_k;
  int mask_kind;
  const void* mask;            // element (b,h,i,j) at b*m_sb + h*m_sh + i*m_sq + j
  int64_t m_sb, m_sh, m_sq;    // 0 on broadcast dims
  const uint8_t* flags;        // bool masks: tile classes
  const unsigned* mask_any_false;  // bool masks: the classify kernel's word, 0 when every element is True
  int64_t f_sb, f_sh, f_sq;    // strides of the flag array (0 on broadcast dims)
  int causal;
  int f16;           // MMA operand type: 0 bf16, 1 fp16 (v's dtype; q/k of 16 bits have it too)
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  int B, H, Sq, Skv, nQt, nKt;
  int Hkv, group;                 // K/V heads; query heads per K/V head (H / Hkv)
  unsigned* status;               // device status word
  unsigned long long* counters;   // device counters
  long long wait_budget;          // clock64 cycles per bounded wait
};

struct FwdParams {
  Common c;
  CUtensorMap tmap_v;  // V as a 4-D tiled map, 128B swizzle, box 64 x 128 keys
  CUtensorMap tmap_q;  // raw q / k rows (16-bit only; see qk_tma)
  CUtensorMap tmap_k;
  int v_s_first;       // map dims are (d, s, h, b) instead of (d, h, s, b)
  int q_s_first, k_s_first;
  int qk_tma;          // 1: q and k are 16-bit and staged by TMA, normalised in place
  CUtensorMap tmap_qp; // the workspace's Q' rows ([B, Sq, H, D], operand type), 128-row boxes (TMA store)
  int save_qp;         // 1: the CTA stores its Q' tiles there for the backward
  float* dq_zero;      // the backward's fp32 dQ' accumulator [B, Sq, H, D], zeroed here (or null)
  CUtensorMap tmap_kc; // the workspace's K' tiles ([B, Skv, Hkv, D], operand type), 128-row boxes
  uint32_t* kflags;    // [B, Hkv, nKt]: 1 once K' of the tile is in tmap_kc's buffer (zeroed per call)
  int kcache;          // 1: K' tiles are shared between CTAs through that buffer
  void* o;
  int64_t o_sb, o_ss, o_sh;
  int o_dt;
  float* lse;  // [B, H, Sq]
};

struct BwdParams {
  Common c;
  CUtensorMap tmap_v;   // V rows, as in FwdParams
  CUtensorMap tmap_do;  // dO rows, 128-row boxes
  CUtensorMap tmap_q;   // Q' rows of the workspace ([B, Sq, H, D], operand type), 64-row boxes
  CUtensorMap tmap_k;   // raw k rows, 128-row boxes (16-bit: 64 columns; fp32: 32 columns, epilogue only)
  CUtensorMap tmap_tab_k;  // the fp32 (cos, sin) table of the keys as [Bt_k * Skv, 128] floats, 32 x 128 boxes
  CUtensorMap tmap_dv;     // dv rows, 128-row boxes (TMA store of the epilogue)
  CUtensorMap tmap_dk;     // dk rows, 128-row boxes (16-bit k only)
  CUtensorMap tmap_dq;  // dq_acc as (d, h, s, b), fp32, 128B swizzle, box 32 x 64 rows (reduce target)
  CUtensorMap tmap_kc;  // the forward's shared K' tiles, 128-row boxes (kp_ready)
  int kp_ready;         // 1: the workspace holds the forward's K' tiles and their flags (a reusing backward)
  const uint32_t* kflags;  // [B, Hkv, nKt]: 1 where the forward published the tile
  int v_s_first, do_s_first, q_s_first, k_s_first, dv_s_first, dk_s_first;
  int qk_tma;
  const void* dout;
  int64_t do_sb, do_ss, do_sh;
  const float* lse;    // [B, H, Sq]
  const float* delta;  // [B, H, Sq]
  float* dq_acc;       // [B, Sq, H, D] fp32, zeroed: scale * dS K' (gradient of the rotated, normed q)
                       // (TMA reduce target through tmap_dq)
  void* dv;
  int64_t dv_sb, dv_ss, dv_sh;
  int dv_dt;
  void* dk;            // dk, finished in the kernel's epilogue (inverse rotation + RMSNorm backward)
  int64_t dk_sb, dk_ss, dk_sh;
  int dk_dt;
  float* dwk_part;     // [B, Hkv, nKt, 4, D]: partial sums of the k norm-weight gradient per CTA and row quarter
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float f16_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w))); }
__device__ __forceinline__ float f16_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The 16-bit operand type of the tensor-core MMAs: bf16 (F16 = false) or fp16
// (F16 = true). Element 2i of a packed word is in its low half.
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t w) {
  if constexpr (F16) return f16_lo(w);
  else return bf16_lo(w);
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t w) {
  if constexpr (F16) return f16_hi(w);
  else return bf16_hi(w);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if constexpr (F16) return pack_f16(lo, hi);
  else return pack_bf16(lo, hi);
}

__device__ __forceinline__ void zero_row(uint8_t* tile, int row, uint32_t half = kHalfBytes) {
#pragma unroll
  for (int c = 0; c < kD / 8; ++c)
    *reinterpret_cast<uint4*>(tile + (c >> 3) * half + sw128_off(row, c & 7)) = make_uint4(0, 0, 0, 0);
}

// Two floats as a packed word of a 16-bit row type (kDtBF16 or kDtF16).
__device__ __forceinline__ uint32_t pack_dt(int dt, float lo, float hi) {
  return dt == kDtF16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}

// Stores elements [32*q4, 32*q4 + 32) of a row to a bf16, fp16 or fp32
// destination (dt).
__device__ __forceinline__ void store_chunk32(void* base, int64_t off, int dt, int q4, const float (&y)[32]) {
  if (dt == kDtF32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off) + 8 * q4;
#pragma unroll
    for (int c = 0; c < 8; ++c) p[c] = make_float4(y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]);
  } else {
    uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + off) + 4 * q4;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      p[c] = make_uint4(pack_dt(dt, y[8 * c], y[8 * c + 1]), pack_dt(dt, y[8 * c + 2], y[8 * c + 3]),
                        pack_dt(dt, y[8 * c + 4], y[8 * c + 5]), pack_dt(dt, y[8 * c + 6], y[8 * c + 7]));
  }
}

// Loads elements [8c, 8c+8) of the row at element offset `off` (bf16, fp16
// or fp32 source, dt).
__device__ __forceinline__ void load_chunk8(const void* base, int64_t off, int dt, int c, float (&v)[8]) {
  if (dt == kDtF32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off) + 2 * c;
    const float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off) + c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = dt == kDtF16 ? f16_lo(w[e]) : bf16_lo(w[e]);
      v[2 * e + 1] = dt == kDtF16 ? f16_hi(w[e]) : bf16_hi(w[e]);
    }
  }
}

// Bounded wait on an mbarrier phase that also gives up when another role of
// the CTA has aborted; a wait that runs out of budget raises the CTA's abort
// flag.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// As wait_bar, acquiring at cluster scope (barriers with remote arrivals).
__device__ __forceinline__ bool wait_bar_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                 long long budget) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// Warp-uniform forms: every lane waits, and the warp proceeds only if all of
// them succeeded, so that warp-collective instructions (tcgen05.ld/st,
// shuffles) that follow are never reached by part of a warp.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              long long budget) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, budget));
}
__device__ __forceinline__ bool wait_bar_cluster_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                      long long budget) {
  return __all_sync(0xffffffffu, wait_bar_cluster(bar, parity, abort_flag, budget));
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads: the
// result is the same in every thread (a uniform exit decision).
__device__ __forceinline__ bool named_bar_any(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// max(a, b, c) in one instruction (three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x on the MUFU unit (flushes denormal results to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Kernels of a call are chained with programmatic dependent launch: a kernel
// may be scheduled while its predecessor on the stream finishes, and waits
// here, before its first global-memory access, until that predecessor has
// completed and its writes are visible (a no-op when launched without it).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches `kern` with the programmatic-stream-serialisation attribute (see
// grid_dependency_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ void record_timeout(const Common& c) {
  atomicOr(c.status, kStatusTimeout);
  atomicAdd(c.counters + kCtrTimeouts, 1ull);
}

}  // namespace st
