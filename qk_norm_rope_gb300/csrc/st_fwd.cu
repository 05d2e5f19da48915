// Forward kernel: fused RMSNorm + RoPE prologue, tcgen05 QK^T and PV with
// TMEM accumulators, online base-2 softmax, O and log-sum-exp epilogue.
//
// One CTA per (pair of 128-row query tiles, head, batch), warp-specialised:
//   warps 0-7   softmax: warp w serves query tile w/4 and TMEM lanes
//               32*(w%4).. (one thread per query row); two passes over the
//               row's 128 scores in TMEM: the max of the raw scores, then
//               P = exp2(s*scale*log2e - max) with the scale folded into one FMA
//   warps 8-15  operand prologue, two lanes per row (one per 64-column half):
//               Q' for both query tiles, then K' for every key tile of a
//               kStages-deep ring; bf16 rows arrive by TMA in the operand
//               layout and are normalised and rotated in place, their (cos,
//               sin) rows being fetched while the TMA is in flight (fp32 rows
//               are read from global memory, one thread per row)
//   warp 16     TMEM allocation + tcgen05.mma issue (one thread)
//   warp 17     TMA: raw Q and K rows, V tiles
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each; P_i (bf16)
// overwrites the first 64 columns of S_i and feeds PV from TMEM.
// MMA issue order per key tile n: PV0(n-1), S0(n), PV1(n-1), S1(n), so that
// while one softmax group works on its scores the tensor core computes the
// other's.
#include "st_common.cuh"
#include "st_kernels.h"
#include "st_prologue.cuh"

namespace st {

namespace {

constexpr int kStages = 2;
constexpr int kSoftWarps = 8;
constexpr int kWarpProl0 = 8, kProlWarps = 8;
constexpr int kWarpMma = 16, kWarpTma = 17;
constexpr int kFwdWarps = 18;
constexpr int kFwdThreads = kFwdWarps * 32;
// rescale O only when the running max grows by more than 8 (base 2); exact
// either way since O and l always share the same reference max
constexpr float kRescaleThreshold = 8.0f;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;                                  // 2 tiles
constexpr uint32_t kOffK = 2 * kTileBytes;                     // kStages tiles
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;       // kStages tiles
constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;
constexpr uint32_t kOffW = kOffBar + 256;                      // q and k norm weights, fp32
constexpr uint32_t kFwdSmem = kOffW + 2 * kD * 4 + 1024;

enum {
  kBarQRaw = 0,                       // raw q rows landed (TMA)
  kBarQFull,                          // Q' ready (prologue)
  kBarKRaw,                           // + stage: raw k rows landed (TMA)
  kBarKFull = kBarKRaw + kStages,     // + stage: K' ready (prologue)
  kBarVFull = kBarKFull + kStages,    // + stage
  kBarKVEmpty = kBarVFull + kStages,  // + stage
  kBarSFull = kBarKVEmpty + kStages,  // + tile (0/1)
  kBarPFull = kBarSFull + 2,          // + tile, 256 arrivals
  kBarOFull = kBarPFull + 2,
  kNumBars = kBarOFull + 1
};

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, kHalfBytes, 1024);
}

template <int MK>
__device__ __forceinline__ uint8_t tile_flag(const Common& c, int b, int h, int qt, int kt) {
  if (qt >= c.nQt) return kTileAllFalse;
  if constexpr (MK == kMaskBool) return c.flags[b * c.f_sb + h * c.f_sh + qt * c.f_sq + kt];
  if constexpr (MK == kMaskNone) return kTileAllTrue;
  return kTileMixed;  // additive masks are always applied
}

__device__ __forceinline__ float c_wq(const Common& c, int d) { return __ldg(c.wq + d); }
__device__ __forceinline__ float c_wk(const Common& c, int d) { return __ldg(c.wk + d); }

// Next key tile at or after kt that at least one of the two query tiles needs.
template <int MK>
__device__ __forceinline__ int next_tile(const Common& c, int b, int h, int qt0, int kt, int kt_end) {
  if constexpr (MK != kMaskBool) return kt;
  for (; kt < kt_end; ++kt)
    if (tile_flag<MK>(c, b, h, qt0, kt) != kTileAllFalse || tile_flag<MK>(c, b, h, qt0 + 1, kt) != kTileAllFalse) break;
  return kt;
}

// Base-2 scores of 32 key columns [j0, j0 + 32) of query row i from their raw
// TMEM values: s * scale * log2(e) (+ mask * log2(e)), -inf where a bool mask
// is False, beyond the causal diagonal or at keys >= S_kv. Tiles that need no
// masking take the caller's fast path instead.
// Additive-mask rows are read as 16-byte vectors when the mask's base and
// strides allow it (and the chunk lies inside the row), all issued before the
// first use and pinned so that they complete together.
template <int MK, bool CAUSAL>
__device__ __forceinline__ void masked_scores32(const Common& c, const uint32_t (&raw)[32], int b, int h, int i,
                                                int j0, uint8_t flag, uint32_t mbits, float (&s)[32],
                                                bool mask_vec, uint32_t* scratch) {
#pragma unroll
  for (int t = 0; t < 32; ++t) s[t] = __uint_as_float(raw[t]) * c.scale_log2;
  if (flag == kTileAllFalse) {
#pragma unroll
    for (int t = 0; t < 32; ++t) s[t] = -INFINITY;
    return;
  }
  if constexpr (MK == kMaskBool) {
    if (flag == kTileMixed) {
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if (!((mbits >> t) & 1u)) s[t] = -INFINITY;
    }
  } else if constexpr (MK == kMaskF32) {
    if (i < c.Sq) {
      const float* mrow = static_cast<const float*>(c.mask) + b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j0;
      if (mask_vec && j0 + 32 <= c.Skv) {
        uint4 u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) u[k] = ldg_nc_v4(mrow + 4 * k);
        uint32_t folded = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) folded ^= u[k].x ^ u[k].y ^ u[k].z ^ u[k].w;
        pin_loads(folded, scratch);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          s[4 * k] = fmaf(__uint_as_float(u[k].x), kLog2e, s[4 * k]);
          s[4 * k + 1] = fmaf(__uint_as_float(u[k].y), kLog2e, s[4 * k + 1]);
          s[4 * k + 2] = fmaf(__uint_as_float(u[k].z), kLog2e, s[4 * k + 2]);
          s[4 * k + 3] = fmaf(__uint_as_float(u[k].w), kLog2e, s[4 * k + 3]);
        }
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (j0 + t < c.Skv) s[t] = fmaf(__ldg(mrow + t), kLog2e, s[t]);
      }
    }
  } else if constexpr (MK == kMaskBF16) {
    if (i < c.Sq) {
      const __nv_bfloat16* mrow =
          static_cast<const __nv_bfloat16*>(c.mask) + b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j0;
      if (mask_vec && j0 + 32 <= c.Skv) {
        uint4 u[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) u[k] = ldg_nc_v4(mrow + 8 * k);
        uint32_t folded = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) folded ^= u[k].x ^ u[k].y ^ u[k].z ^ u[k].w;
        pin_loads(folded, scratch);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            s[8 * k + 2 * e] = fmaf(bf16_lo(w[e]), kLog2e, s[8 * k + 2 * e]);
            s[8 * k + 2 * e + 1] = fmaf(bf16_hi(w[e]), kLog2e, s[8 * k + 2 * e + 1]);
          }
        }
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (j0 + t < c.Skv) s[t] = fmaf(__bfloat162float(mrow[t]), kLog2e, s[t]);
      }
    }
  }
  if constexpr (CAUSAL) {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (j0 + t > i) s[t] = -INFINITY;
  }
  if (j0 + 32 > c.Skv) {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (j0 + t >= c.Skv) s[t] = -INFINITY;
  }
}

template <int MK, bool CAUSAL, bool QKT>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const Common& c = P.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
  const int pair = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int qt0 = 2 * pair;

  if (warp == kWarpMma) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars[kBarQRaw], 1);
    mbar_init(&bars[kBarQFull], kProlWarps * 32);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kBarKRaw + s], 1);
      mbar_init(&bars[kBarKFull + s], kProlWarps * 32);
      mbar_init(&bars[kBarVFull + s], 1);
      mbar_init(&bars[kBarKVEmpty + s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[kBarSFull + t], 1);
      mbar_init(&bars[kBarPFull + t], 128);
    }
    mbar_init(&bars[kBarOFull], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  float* sW = reinterpret_cast<float*>(sm + kOffW);  // [wq | wk]
  if (tid < 2 * kD) sW[tid] = tid < kD ? c_wq(P.c, tid) : c_wk(P.c, tid - kD);
  if (warp == kWarpTma && lane_id == 0) {
    tma_prefetch_desc(&P.tmap_v);
    if constexpr (QKT) {
      tma_prefetch_desc(&P.tmap_q);
      tma_prefetch_desc(&P.tmap_k);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  int kt_end = c.nKt;
  if (CAUSAL) kt_end = min(c.nKt, (qt0 * kTile + 2 * kTile - 1) / kTile + 1);
  const long long budget = c.wait_budget;

  if (warp < kSoftWarps) {
    // ------------------------------------------------------------ softmax
    const int ti = warp >> 2;                 // query tile of the pair
    const int r = (warp & 3) * 32 + lane_id;  // row within the tile = TMEM lane
    const int i = (qt0 + ti) * kTile + r;
    const uint32_t lane = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + ti * 128 + lane, tO = tmem + 256 + ti * 128 + lane;
    const float sc = c.scale_log2;
    uint32_t* scratch = tslot + 2;  // sink for pin_loads
    constexpr int kVecElems = MK == kMaskBF16 ? 8 : 4;  // elements per 16 bytes
    const bool mask_vec = (reinterpret_cast<uintptr_t>(c.mask) & 15u) == 0 && c.m_sb % kVecElems == 0 &&
                          c.m_sh % kVecElems == 0 && c.m_sq % kVecElems == 0;
    float m_run = -INFINITY, l_run = 0.f;
    int n = 0, useful = 0;
    bool ok = true;
    for (int kt = next_tile<MK>(c, b, h, qt0, 0, kt_end); kt < kt_end; kt = next_tile<MK>(c, b, h, qt0, kt + 1, kt_end), ++n) {
      const uint8_t flag = tile_flag<MK>(c, b, h, qt0 + ti, kt);
      useful += (flag != kTileAllFalse && (!CAUSAL || kt <= qt0 + ti)) ? 1 : 0;
      const int j0 = kt * kTile;
      // plain tiles: no mask values, no causal diagonal, no key bound inside
      const bool plain = (flag == kTileAllTrue || (MK == kMaskNone && flag != kTileAllFalse)) &&
                         (!CAUSAL || j0 + kTile - 1 <= (qt0 + ti) * kTile) && j0 + kTile <= c.Skv;
      uint32_t mbits[4] = {~0u, ~0u, ~0u, ~0u};
      if (MK == kMaskBool && flag == kTileMixed && i < c.Sq) {
        const uint8_t* mrow = static_cast<const uint8_t*>(c.mask) + b * c.m_sb + h * c.m_sh + (int64_t)i * c.m_sq + j0;
        const int nvalid = min(kTile, c.Skv - j0);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t bits = 0;
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (32 * q4 + t < nvalid && __ldg(mrow + 32 * q4 + t)) bits |= 1u << t;
          mbits[q4] = bits;
        }
      }
      if (!(ok = wait_bar_warp(&bars[kBarSFull + ti], n & 1, abort_flag, budget))) break;
      tc_fence_after();
      // pass 1: row max (raw scores on plain tiles; the scale is positive)
      float mt = -INFINITY;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t raw[32];
        tmem_ld32(tS + 32 * q4, raw);
        if (plain) {
          float m0 = __uint_as_float(raw[0]), m1 = __uint_as_float(raw[1]);
#pragma unroll
          for (int t = 2; t < 32; t += 2) {
            m0 = fmaxf(m0, __uint_as_float(raw[t]));
            m1 = fmaxf(m1, __uint_as_float(raw[t + 1]));
          }
          mt = fmaxf(mt, fmaxf(m0, m1) * sc);
        } else {
          // scaled and masked once; pass 2 reads them back instead of the mask
          float sv[32];
          masked_scores32<MK, CAUSAL>(c, raw, b, h, i, j0 + 32 * q4, flag, mbits[q4], sv, mask_vec, scratch);
          uint32_t w32[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            mt = fmaxf(mt, sv[t]);
            w32[t] = __float_as_uint(sv[t]);
          }
          tmem_st32(tS + 32 * q4, w32);
        }
      }
      if (!plain) tmem_st_wait();
      float corr = 1.f;
      if (mt > m_run + kRescaleThreshold || (m_run == -INFINITY && mt > -INFINITY)) {
        corr = ex2(m_run - mt);  // 0 when m_run is -inf
        m_run = mt;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // pass 2: P = exp2(s - m) (bf16 into the first 64 S columns), row sum
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t raw[32], pw[16];
        tmem_ld32(tS + 32 * q4, raw);
        if (plain) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float p0 = ex2(fmaf(__uint_as_float(raw[2 * t]), sc, -m_use));
            const float p1 = ex2(fmaf(__uint_as_float(raw[2 * t + 1]), sc, -m_use));
            ls0 += p0;
            ls1 += p1;
            pw[t] = pack_bf16(p0, p1);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float p0 = ex2(__uint_as_float(raw[2 * t]) - m_use), p1 = ex2(__uint_as_float(raw[2 * t + 1]) - m_use);
            ls0 += p0;
            ls1 += p1;
            pw[t] = pack_bf16(p0, p1);
          }
        }
        tmem_st16(tS + 16 * q4, pw);
      }
      l_run = l_run * corr + (ls0 + ls1);
      if (n > 0 && __any_sync(0xffffffffu, corr != 1.f)) {  // warp-uniform: tcgen05.ld/st are collective
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t r32[32];
          tmem_ld32(tO + 32 * q4, r32);
#pragma unroll
          for (int t = 0; t < 32; ++t) r32[t] = __float_as_uint(__uint_as_float(r32[t]) * corr);
          tmem_st32(tO + 32 * q4, r32);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kBarPFull + ti]);
    }
    // ---- epilogue: O / l, LSE
    if (ok && n > 0) ok = wait_bar_warp(&bars[kBarOFull], 0, abort_flag, budget);
    if (ok) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const int64_t ooff = b * P.o_sb + (int64_t)i * P.o_ss + h * P.o_sh;
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t r32[32];
        if (n > 0) {
          tmem_ld32(tO + 32 * q4, r32);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) r32[t] = 0u;
        }
        float y[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) y[t] = __uint_as_float(r32[t]) * inv;
        if (i < c.Sq) store_chunk32(P.o, ooff, P.o_f32, q4, y);
      }
      if (i < c.Sq)
        P.lse[((int64_t)b * c.H + h) * c.Sq + i] = (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      if (r == 0 && qt0 + ti < c.nQt) {  // key tiles this query tile skipped or found fully masked
        atomicAdd(c.counters + kCtrTilesSkipped, (unsigned long long)(c.nKt - useful));
        atomicAdd(c.counters + kCtrTilesTotal, (unsigned long long)c.nKt);
      }
    }
  } else if (warp < kWarpProl0 + kProlWarps) {
    // ------------------------------------------------------------ operand prologue
    const int p = tid - kWarpProl0 * 32;                      // 0..255
    const int prow = (p >> 5) * 16 + (lane_id & 15), hh = lane_id >> 4;  // TMA path: half-row
    bool ok = true;
    if constexpr (QKT) ok = wait_bar_warp(&bars[kBarQRaw], 0, abort_flag, budget);
    if (ok) {
#pragma unroll 1
      for (int ti = 0; ti < 2; ++ti) {
        uint8_t* tile = sm + kOffQ + ti * kTileBytes;
        if constexpr (QKT) {
          const int i = (qt0 + ti) * kTile + prow;  // rows past S_q stay TMA zeros
          HalfRowPrologue hp;
          if (i < c.Sq) {
            const __half2* t16 = c.tab16_q + b * c.tab_q_sb + (int64_t)i * kPairs;
            hp.prefetch(t16, hh);
            hp.prefetch2(t16, hh);
          }
          hp.finish(tile, prow, hh, sW, c.eps, i < c.Sq);
        } else if (p < kTile) {
          const int i = (qt0 + ti) * kTile + p;
          if (i < c.Sq)
            rope_norm_global(c.q.p, b * c.q.sb + (int64_t)i * c.q.ss + h * c.q.sh, c.q.is_f32, c.wq, c.eps,
                             c.tab_q + b * c.tab_q_sb + (int64_t)i * kPairs, tile, p);
          else
            zero_row(tile, p);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[kBarQFull]);
    }
    int n = 0;
    for (int kt = next_tile<MK>(c, b, h, qt0, 0, kt_end); ok && kt < kt_end;
         kt = next_tile<MK>(c, b, h, qt0, kt + 1, kt_end), ++n) {
      const int slot = n % kStages;
      uint8_t* tile = sm + kOffK + slot * kTileBytes;
      if constexpr (QKT) {
        const int j = kt * kTile + prow;
        HalfRowPrologue hp;
        if (j < c.Skv) {
          const __half2* t16 = c.tab16_k + b * c.tab_k_sb + (int64_t)j * kPairs;
          hp.prefetch(t16, hh);
          hp.prefetch2(t16, hh);
        }
        if (!wait_bar_warp(&bars[kBarKRaw + slot], (n / kStages) & 1, abort_flag, budget)) break;
        hp.finish(tile, prow, hh, sW + kD, c.eps, j < c.Skv);
      } else {
        if (n >= kStages && !wait_bar(&bars[kBarKVEmpty + slot], ((n / kStages) - 1) & 1, abort_flag, budget)) break;
        if (p < kTile) {
          const int j = kt * kTile + p;
          if (j < c.Skv)
            rope_norm_global(c.k.p, b * c.k.sb + (int64_t)j * c.k.ss + h * c.k.sh, c.k.is_f32, c.wk, c.eps,
                             c.tab_k + b * c.tab_k_sb + (int64_t)j * kPairs, tile, p);
          else
            zero_row(tile, p);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[kBarKFull + slot]);
    }
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA: raw Q, raw K, V
    if (lane_id == 0) {
      if constexpr (QKT) {
        mbar_arrive_expect_tx(&bars[kBarQRaw], 2 * kTileBytes);
#pragma unroll 1
        for (int ti = 0; ti < 2; ++ti) {
          const int row = (qt0 + ti) * kTile;
          const int y = P.q_s_first ? row : h, z = P.q_s_first ? h : row;
          uint8_t* tile = sm + kOffQ + ti * kTileBytes;
          tma_load_4d(tile, &P.tmap_q, &bars[kBarQRaw], 0, y, z, b);
          tma_load_4d(tile + kHalfBytes, &P.tmap_q, &bars[kBarQRaw], 64, y, z, b);
        }
      }
      int n = 0;
      for (int kt = next_tile<MK>(c, b, h, qt0, 0, kt_end); kt < kt_end;
           kt = next_tile<MK>(c, b, h, qt0, kt + 1, kt_end), ++n) {
        const int slot = n % kStages;
        if (n >= kStages && !wait_bar(&bars[kBarKVEmpty + slot], ((n / kStages) - 1) & 1, abort_flag, budget)) break;
        if constexpr (QKT) {
          uint8_t* ktile = sm + kOffK + slot * kTileBytes;
          const int y = P.k_s_first ? kt * kTile : h, z = P.k_s_first ? h : kt * kTile;
          mbar_arrive_expect_tx(&bars[kBarKRaw + slot], kTileBytes);
          tma_load_4d(ktile, &P.tmap_k, &bars[kBarKRaw + slot], 0, y, z, b);
          tma_load_4d(ktile + kHalfBytes, &P.tmap_k, &bars[kBarKRaw + slot], 64, y, z, b);
        }
        uint8_t* tile = sm + kOffV + slot * kTileBytes;
        const int y = P.v_s_first ? kt * kTile : h, z = P.v_s_first ? h : kt * kTile;
        mbar_arrive_expect_tx(&bars[kBarVFull + slot], kTileBytes);
        tma_load_4d(tile, &P.tmap_v, &bars[kBarVFull + slot], 0, y, z, b);
        tma_load_4d(tile + kHalfBytes, &P.tmap_v, &bars[kBarVFull + slot], 64, y, z, b);
      }
      // every issued load lands before the CTA exits
      // (these waits do not give up on abort; each is bounded)
      if constexpr (QKT) mbar_wait(&bars[kBarQRaw], 0, budget);
      for (int m = max(0, n - kStages); m < n; ++m) {
        mbar_wait(&bars[kBarVFull + m % kStages], (m / kStages) & 1, budget);
        if constexpr (QKT) mbar_wait(&bars[kBarKRaw + m % kStages], (m / kStages) & 1, budget);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue
    if (lane_id == 0) {
      const uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(128, 128, 0, 1);
      const uint32_t aQ0 = smem_u32(sm + kOffQ), aQ1 = aQ0 + kTileBytes;
      const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
      bool ok = wait_bar(&bars[kBarQFull], 0, abort_flag, budget);
      int kt = next_tile<MK>(c, b, h, qt0, 0, kt_end);
      int n = 0;
      bool issued = false;
      if (ok && kt < kt_end) {
        ok = wait_bar(&bars[kBarKFull + 0], 0, abort_flag, budget);
        if (ok) {
          tc_fence_after();
          const uint32_t aK = smem_u32(sm + kOffK);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS0, kmajor_desc(aQ0, kk), kmajor_desc(aK, kk), idesc_qk, kk > 0);
          mma_commit(&bars[kBarSFull + 0]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS1, kmajor_desc(aQ1, kk), kmajor_desc(aK, kk), idesc_qk, kk > 0);
          mma_commit(&bars[kBarSFull + 1]);
          issued = true;
        }
      }
      while (ok && kt < kt_end) {
        const int slot = n % kStages;
        const int kt_next = next_tile<MK>(c, b, h, qt0, kt + 1, kt_end);
        const bool has_next = kt_next < kt_end;
        const int nslot = (n + 1) % kStages;
        const uint32_t aV = smem_u32(sm + kOffV + slot * kTileBytes);
        if (!(ok = wait_bar(&bars[kBarVFull + slot], (n / kStages) & 1, abort_flag, budget))) break;
        if (!(ok = wait_bar(&bars[kBarPFull + 0], n & 1, abort_flag, budget))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts(tO0, tS0 + kk * 8, mnmajor_desc(aV, kk), idesc_pv, (n > 0 || kk > 0));
        if (has_next) {
          if (!(ok = wait_bar(&bars[kBarKFull + nslot], ((n + 1) / kStages) & 1, abort_flag, budget))) break;
          tc_fence_after();
          const uint32_t aK = smem_u32(sm + kOffK + nslot * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS0, kmajor_desc(aQ0, kk), kmajor_desc(aK, kk), idesc_qk, kk > 0);
          mma_commit(&bars[kBarSFull + 0]);
        }
        if (!(ok = wait_bar(&bars[kBarPFull + 1], n & 1, abort_flag, budget))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts(tO1, tS1 + kk * 8, mnmajor_desc(aV, kk), idesc_pv, (n > 0 || kk > 0));
        mma_commit(&bars[kBarKVEmpty + slot]);
        if (has_next) {
          const uint32_t aK = smem_u32(sm + kOffK + nslot * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS1, kmajor_desc(aQ1, kk), kmajor_desc(aK, kk), idesc_qk, kk > 0);
          mma_commit(&bars[kBarSFull + 1]);
        }
        kt = kt_next;
        ++n;
      }
      if (issued) {
        // every MMA done (also on abort) before anyone reads O or frees TMEM
        mma_commit(&bars[kBarOFull]);
        if (!ok) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&bars[kBarOFull], 0) && clock64() - t0 < budget) {
          }
        }
      }
    }
  }

  if (*abort_flag && tid == 0) record_timeout(c);
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int MK, bool CAUSAL, bool QKT>
cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_kernel<MK, CAUSAL, QKT>;
  static unsigned configured = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured & (1u << (dev & 31)))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e != cudaSuccess) return e;
    configured |= 1u << (dev & 31);
  }
  dim3 grid((p.c.nQt + 1) / 2, p.c.H, p.c.B);
  kern<<<grid, kFwdThreads, kFwdSmem, stream>>>(p);
  return cudaGetLastError();
}

template <bool QKT>
cudaError_t launch_fwd_q(const FwdParams& p, cudaStream_t stream) {
  if (p.c.causal) return launch_fwd_t<kMaskNone, true, QKT>(p, stream);  // masks and causal never combine
  switch (p.c.mask_kind) {
    case kMaskBool: return launch_fwd_t<kMaskBool, false, QKT>(p, stream);
    case kMaskF32: return launch_fwd_t<kMaskF32, false, QKT>(p, stream);
    case kMaskBF16: return launch_fwd_t<kMaskBF16, false, QKT>(p, stream);
    default: return launch_fwd_t<kMaskNone, false, QKT>(p, stream);
  }
}

// Kernels are specialised on the mask kind, causal masking and whether q/k
// are staged by TMA, so that each carries only its own code.
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  return p.qk_tma ? launch_fwd_q<true>(p, stream) : launch_fwd_q<false>(p, stream);
}

}  // namespace st
