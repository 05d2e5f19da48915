// Backward main kernel: one CTA per (key tile of 128 rows, head, batch),
// 128 threads, thread t owns key row t (TMEM lane t). Per query tile:
//   prologue  Q' = RoPE(RMSNorm(q)) and dO into 128B-swizzled tiles;
//   MMA 1/2   S^T = K' Q'^T and dP^T = V dO^T into TMEM;
//   SIMT      P^T = exp2(S^T * scale*log2e - LSE*log2e) (mask / causal /
//             bounds applied), dS^T = P^T (dP^T - Delta); P^T goes back to
//             TMEM (A operand of MMA 3), dS^T to shared memory;
//   MMA 3/4/5 dV += P^T dO, dK' += dS^T Q', dQ = dS K' (TMEM);
//   dQ rows   scaled and added atomically into the fp32 dQ accumulator.
// Epilogue: dV out; dK' scaled, inverse-rotated and pushed through the
// RMSNorm backward; per-CTA partial sums of the k-norm weight gradient.
#include "st_common.cuh"
#include "st_kernels.h"

namespace st {

namespace {

constexpr int kBwdThreads = 128;
constexpr uint32_t kBwdSmem = 5 * kTileBytes + 2 * 512 + 1024 + 1024;

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, kHalfBytes, 1024);
}

// Mask value (base-2 units, -inf for masked) for query row i, key j.
__device__ __forceinline__ float mask_term(const Common& c, int b, int h, int i, int j) {
  const int64_t off = b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j;
  if (c.mask_kind == kMaskBool) return __ldg(static_cast<const uint8_t*>(c.mask) + off) ? 0.f : -INFINITY;
  if (c.mask_kind == kMaskF32) return __ldg(static_cast<const float*>(c.mask) + off) * kLog2e;
  return __bfloat162float(static_cast<const __nv_bfloat16*>(c.mask)[off]) * kLog2e;
}

__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(const __grid_constant__ BwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm;
  uint8_t* sV = sm + kTileBytes;
  uint8_t* sQ = sm + 2 * kTileBytes;
  uint8_t* sdO = sm + 3 * kTileBytes;
  uint8_t* sdS = sm + 4 * kTileBytes;
  float* sLse = reinterpret_cast<float*>(sm + 5 * kTileBytes);
  float* sDelta = sLse + 128;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sDelta + 128);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);

  const Common& c = P.c;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int j = kt * kTile + tid;  // this thread's key row

  if (warp == 0) {
    tmem_alloc(tslot, 512);
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
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;

  if (j < c.Skv) {
    float x[kD];
    load_row(c.k.p, b * c.k.sb + (int64_t)j * c.k.ss + h * c.k.sh, c.k.is_f32, x);
    norm_rope_store(x, c.wk, c.eps, c.tab_k + b * c.tab_k_sb + (int64_t)j * kPairs, sK, tid);
    copy_row_bf16(c.v.p, b * c.v.sb + (int64_t)j * c.v.ss + h * c.v.sh, sV, tid);
  } else {
    zero_row(sK, tid);
    zero_row(sV, tid);
  }

  const int qt_begin = c.causal ? min(c.nQt, (kt * kTile) / kTile) : 0;
  const uint32_t idesc_kk = idesc_bf16(128, 128, 0, 0);
  const uint32_t idesc_kmn = idesc_bf16(128, 128, 0, 1);
  const uint32_t idesc_mnmn = idesc_bf16(128, 128, 1, 1);
  const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), adO = smem_u32(sdO), adS = smem_u32(sdS);

  uint32_t phase = 0;
  bool first = true, failed = false;
  int skipped = qt_begin;

  for (int qt = qt_begin; qt < c.nQt; ++qt) {
    uint8_t flag = kTileMixed;
    if (c.mask_kind == kMaskBool) flag = c.flags[b * c.f_sb + h * c.f_sh + qt * c.f_sq + kt];
    if (flag == kTileAllFalse) {
      ++skipped;
      continue;
    }
    const int i = qt * kTile + tid;  // query row loaded by this thread
    if (i < c.Sq) {
      float x[kD];
      load_row(c.q.p, b * c.q.sb + (int64_t)i * c.q.ss + h * c.q.sh, c.q.is_f32, x);
      norm_rope_store(x, c.wq, c.eps, c.tab_q + b * c.tab_q_sb + (int64_t)i * kPairs, sQ, tid);
      copy_row_bf16(P.dout, b * P.do_sb + (int64_t)i * P.do_ss + h * P.do_sh, sdO, tid);
      const int64_t r = ((int64_t)b * c.H + h) * c.Sq + i;
      const float lse = P.lse[r];
      sLse[tid] = (lse == -INFINITY) ? INFINITY : lse * kLog2e;  // dead rows give P = 0
      sDelta[tid] = P.delta[r];
    } else {
      zero_row(sQ, tid);
      zero_row(sdO, tid);
      sLse[tid] = INFINITY;
      sDelta[tid] = 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ss(tS, kmajor_desc(aK, kk), kmajor_desc(aQ, kk), idesc_kk, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ss(tdP, kmajor_desc(aV, kk), kmajor_desc(adO, kk), idesc_kk, kk > 0);
      mma_commit(bar);
    }
    __syncwarp();
    bool ok = mbar_wait(bar, phase, c.wait_budget);
    phase ^= 1;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();

    // ---- P^T and dS^T for key row j, query columns qt*128 + cc
    {
      const bool key_ok = j < c.Skv;
      uint32_t r32[32], pw[32];
      float p[kTile];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tS + lane + 32 * q4, r32);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int cc = 32 * q4 + t;
          const int iq = qt * kTile + cc;
          float s2 = __uint_as_float(r32[t]) * c.scale_log2;
          if (c.mask_kind != kMaskNone && iq < c.Sq && key_ok &&
              !(c.mask_kind == kMaskBool && flag == kTileAllTrue))
            s2 += mask_term(c, b, h, iq, j);
          if (c.causal && j > iq) s2 = -INFINITY;
          float pv = exp2f(s2 - sLse[cc]);
          if (!key_ok) pv = 0.f;
          p[cc] = pv;
        }
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int t = 0; t < 32; ++t) pw[t] = pack_bf16(p[64 * hh + 2 * t], p[64 * hh + 2 * t + 1]);
        tmem_st32(tS + lane + 32 * hh, pw);
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tdP + lane + 32 * q4, r32);
#pragma unroll
        for (int t = 0; t < 32; t += 8) {
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c0 = 32 * q4 + t + 2 * u;
            const float d0 = p[c0] * (__uint_as_float(r32[t + 2 * u]) - sDelta[c0]);
            const float d1 = p[c0 + 1] * (__uint_as_float(r32[t + 2 * u + 1]) - sDelta[c0 + 1]);
            w4[u] = pack_bf16(d0, d1);
          }
          const int chunk = (32 * q4 + t) >> 3;  // 0..15
          *reinterpret_cast<uint4*>(sdS + (chunk >> 3) * kHalfBytes + sw128_off(tid, chunk & 7)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t acc = first ? 0u : 1u;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ts(tdV, tS + kk * 8, mnmajor_desc(adO, kk), idesc_kmn, (acc || kk > 0));
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tdK, kmajor_desc(adS, kk), mnmajor_desc(aQ, kk), idesc_kmn, (acc || kk > 0));
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma_ss(tdP, mnmajor_desc(adS, kk), mnmajor_desc(aK, kk), idesc_mnmn, kk > 0);
      mma_commit(bar);
    }
    __syncwarp();
    ok = mbar_wait(bar, phase, c.wait_budget);
    phase ^= 1;
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();

    // ---- dQ rows: lane t holds query row qt*128 + t
    {
      const int iq = qt * kTile + tid;
      uint32_t r32[32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tdP + lane + 32 * q4, r32);
        if (iq < c.Sq) {
          float4* dst = reinterpret_cast<float4*>(P.dq_acc + (((int64_t)b * c.Sq + iq) * c.H + h) * kD + 32 * q4);
#pragma unroll
          for (int t = 0; t < 32; t += 4)
            atomicAdd(dst + t / 4, make_float4(__uint_as_float(r32[t]) * c.scale, __uint_as_float(r32[t + 1]) * c.scale,
                                               __uint_as_float(r32[t + 2]) * c.scale,
                                               __uint_as_float(r32[t + 3]) * c.scale));
        }
      }
    }
    first = false;
  }

  if (failed) {
    if (tid == 0) record_timeout(c);
    mbar_wait(bar, phase ^ 1, c.wait_budget);
  } else {
    // ---- epilogue: dV, dK (inverse RoPE + RMSNorm backward), k-norm weight partials
    float* red = reinterpret_cast<float*>(sQ);  // [128][129] fp32, reuses sQ/sdO/sdS
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    float g[kD];
    uint32_t r32[32];
    if (!first) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tdV + lane + 32 * q4, r32);
#pragma unroll
        for (int t = 0; t < 32; ++t) g[32 * q4 + t] = __uint_as_float(r32[t]);
      }
    } else {
#pragma unroll
      for (int d = 0; d < kD; ++d) g[d] = 0.f;
    }
    if (j < c.Skv) store_row(P.dv, b * P.dv_sb + (int64_t)j * P.dv_ss + h * P.dv_sh, P.dv_f32, g);
    if (!first) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tdK + lane + 32 * q4, r32);
#pragma unroll
        for (int t = 0; t < 32; ++t) g[32 * q4 + t] = __uint_as_float(r32[t]) * c.scale;
      }
    } else {
#pragma unroll
      for (int d = 0; d < kD; ++d) g[d] = 0.f;
    }
    float* my = red + tid * (kD + 1);
    if (j < c.Skv) {
      rope_norm_bwd_row(g, c.k.p, b * c.k.sb + (int64_t)j * c.k.ss + h * c.k.sh, c.k.is_f32,
                        c.tab_k + b * c.tab_k_sb + (int64_t)j * kPairs, c.wk, c.eps, my);
      store_row(P.dk, b * P.dk_sb + (int64_t)j * P.dk_ss + h * P.dk_sh, P.dk_f32, g);
    } else {
      for (int d = 0; d < kD; ++d) my[d] = 0.f;
    }
    __syncthreads();
    {
      float acc = 0.f;
      for (int r = 0; r < kTile; ++r) acc += red[r * (kD + 1) + tid];
      P.dwk_part[(((int64_t)b * c.H + h) * c.nKt + kt) * kD + tid] = acc;
    }
    if (tid == 0) {
      atomicAdd(c.counters + kCtrTilesSkipped, (unsigned long long)skipped);
      atomicAdd(c.counters + kCtrTilesTotal, (unsigned long long)c.nQt);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& p, cudaStream_t stream) {
  static unsigned configured = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured & (1u << (dev & 31)))) {
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
    if (e != cudaSuccess) return e;
    configured |= 1u << (dev & 31);
  }
  dim3 grid(p.c.nKt, p.c.H, p.c.B);
  bwd_kernel<<<grid, kBwdThreads, kBwdSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace st
