// Forward kernel: fused RMSNorm + RoPE prologue, tcgen05 QK^T and PV with
// TMEM accumulators, online base-2 softmax, O and log-sum-exp epilogue.
//
// One CTA per (query tile of 128 rows, head, batch); 128 threads, thread t
// owns query row t of the tile (TMEM lane t). Per key tile:
//   1. every thread normalises + rotates one key row into the K' operand
//      tile and copies one value row into the V tile (both 128B-swizzled);
//   2. one thread issues S = Q' K'^T (8 x tcgen05.mma, K = 16 each) into TMEM;
//   3. each thread reads its S row from TMEM, applies scale, mask / causal /
//      bounds, updates the running max and sum, writes P (bf16) back into the
//      S columns and rescales its O row when the max moved;
//   4. one thread issues O += P V with P read from TMEM.
#include "st_common.cuh"
#include "st_kernels.h"

namespace st {

namespace {

constexpr int kFwdThreads = 128;
constexpr uint32_t kFwdSmem = 3 * kTileBytes + 1024 /*barriers*/ + 1024 /*alignment slack*/;

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, kHalfBytes, 1024);
}

// Adds the mask of keys [j0, j0+128) for query row i to the base-2 scores.
// Keys at or beyond S_kv are set to -inf (and their mask is not read).
__device__ __forceinline__ void apply_mask_row(const Common& c, int b, int h, int i, int j0, uint8_t flag,
                                               float (&s)[kTile]) {
  const int nvalid = min(kTile, c.Skv - j0);
  if (i >= c.Sq) return;  // padding row of the last query tile: nothing to read, nothing stored
  if (c.mask_kind == kMaskBool && flag == kTileMixed) {
    const uint8_t* mrow = static_cast<const uint8_t*>(c.mask) + b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j0;
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj)
      if (jj < nvalid && __ldg(mrow + jj) == 0) s[jj] = -INFINITY;
  } else if (c.mask_kind == kMaskF32) {
    const float* mrow = static_cast<const float*>(c.mask) + b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j0;
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj)
      if (jj < nvalid) s[jj] = fmaf(__ldg(mrow + jj), kLog2e, s[jj]);
  } else if (c.mask_kind == kMaskBF16) {
    const __nv_bfloat16* mrow =
        static_cast<const __nv_bfloat16*>(c.mask) + b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j0;
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj)
      if (jj < nvalid) s[jj] = fmaf(__bfloat162float(mrow[jj]), kLog2e, s[jj]);
  }
  if (nvalid < kTile) {
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj)
      if (jj >= nvalid) s[jj] = -INFINITY;
  }
}

__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;
  uint8_t* sK = sm + kTileBytes;
  uint8_t* sV = sm + 2 * kTileBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 3 * kTileBytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);

  const Common& c = P.c;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int i = qt * kTile + tid;

  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tS = tmem, tO = tmem + 128;

  if (i < c.Sq) {
    float x[kD];
    load_row(c.q.p, b * c.q.sb + (int64_t)i * c.q.ss + h * c.q.sh, c.q.is_f32, x);
    norm_rope_store(x, c.wq, c.eps, c.tab_q + b * c.tab_q_sb + (int64_t)i * kPairs, sQ, tid);
  } else {
    zero_row(sQ, tid);
  }

  int kt_end = c.nKt;
  if (c.causal) kt_end = min(c.nKt, (qt * kTile + kTile - 1) / kTile + 1);

  const uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
  const uint32_t idesc_pv = idesc_bf16(128, 128, 0, 1);
  const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);

  float m_run = -INFINITY, l_run = 0.f;
  uint32_t phase = 0;
  bool any = false;
  bool failed = false;
  int skipped = c.nKt - kt_end;

  for (int kt = 0; kt < kt_end; ++kt) {
    uint8_t flag = kTileMixed;
    if (c.mask_kind == kMaskBool) flag = c.flags[b * c.f_sb + h * c.f_sh + qt * c.f_sq + kt];
    if (flag == kTileAllFalse) {
      ++skipped;
      continue;
    }
    const int j = kt * kTile + tid;
    if (j < c.Skv) {
      float x[kD];
      load_row(c.k.p, b * c.k.sb + (int64_t)j * c.k.ss + h * c.k.sh, c.k.is_f32, x);
      norm_rope_store(x, c.wk, c.eps, c.tab_k + b * c.tab_k_sb + (int64_t)j * kPairs, sK, tid);
      copy_row_bf16(c.v.p, b * c.v.sb + (int64_t)j * c.v.ss + h * c.v.sh, sV, tid);
    } else {
      zero_row(sK, tid);
      zero_row(sV, tid);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ss(tS, kmajor_desc(aQ, kk), kmajor_desc(aK, kk), idesc_qk, kk > 0);
      mma_commit(bar);
    }
    __syncwarp();
    bool ok = mbar_wait(bar, phase, c.wait_budget);
    phase ^= 1;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();

    // ---- online softmax on this thread's row
    float s[kTile];
    {
      uint32_t r32[32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tS + lane + 32 * q4, r32);
#pragma unroll
        for (int t = 0; t < 32; ++t) s[32 * q4 + t] = __uint_as_float(r32[t]) * c.scale_log2;
      }
    }
    apply_mask_row(c, b, h, i, kt * kTile, flag, s);
    if (c.causal) {
#pragma unroll
      for (int jj = 0; jj < kTile; ++jj)
        if (kt * kTile + jj > i) s[jj] = -INFINITY;
    }
    float mt = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj) mt = fmaxf(mt, s[jj]);
    const float m_new = fmaxf(m_run, mt);
    const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
    float lsum = 0.f;
    {
      uint32_t pw[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int jj = 64 * hh + 2 * t;
          const float p0 = (m_new == -INFINITY) ? 0.f : exp2f(s[jj] - m_new);
          const float p1 = (m_new == -INFINITY) ? 0.f : exp2f(s[jj + 1] - m_new);
          lsum += p0 + p1;
          pw[t] = pack_bf16(p0, p1);
        }
        tmem_st32(tS + lane + 32 * hh, pw);
      }
    }
    l_run = l_run * corr + lsum;
    m_run = m_new;
    if (any && __any_sync(0xffffffffu, corr != 1.f)) {  // warp-uniform: tcgen05.ld/st are collective
      uint32_t r32[32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tO + lane + 32 * q4, r32);
#pragma unroll
        for (int t = 0; t < 32; ++t) r32[t] = __float_as_uint(__uint_as_float(r32[t]) * corr);
        tmem_st32(tO + lane + 32 * q4, r32);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ts(tO, tS + kk * 8, mnmajor_desc(aV, kk), idesc_pv, (any || kk > 0) ? 1u : 0u);
      mma_commit(bar);
    }
    __syncwarp();
    ok = mbar_wait(bar, phase, c.wait_budget);
    phase ^= 1;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();
    any = true;
  }

  if (failed) {
    if (tid == 0) record_timeout(c);
    // Give the in-flight MMA one more bounded chance to land before TMEM is freed.
    mbar_wait(bar, phase ^ 1, c.wait_budget);
  } else {
    // ---- epilogue: O / l and the log-sum-exp
    float y[kD];
    if (any) {
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      uint32_t r32[32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tO + lane + 32 * q4, r32);
#pragma unroll
        for (int t = 0; t < 32; ++t) y[32 * q4 + t] = __uint_as_float(r32[t]) * inv;
      }
    } else {
#pragma unroll
      for (int d = 0; d < kD; ++d) y[d] = 0.f;
    }
    if (i < c.Sq) {
      store_row(P.o, b * P.o_sb + (int64_t)i * P.o_ss + h * P.o_sh, P.o_f32, y);
      P.lse[((int64_t)b * c.H + h) * c.Sq + i] = (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    }
    if (tid == 0) {
      atomicAdd(c.counters + kCtrTilesSkipped, (unsigned long long)skipped);
      atomicAdd(c.counters + kCtrTilesTotal, (unsigned long long)c.nKt);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  static unsigned configured = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured & (1u << (dev & 31)))) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e != cudaSuccess) return e;
    configured |= 1u << (dev & 31);
  }
  dim3 grid(p.c.nQt, p.c.H, p.c.B);
  fwd_kernel<<<grid, kFwdThreads, kFwdSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace st
