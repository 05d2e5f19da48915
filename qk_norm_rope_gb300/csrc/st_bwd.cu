// Backward main kernel: one CTA per (key tile of 128 rows, head, batch),
// warp-specialised, looping over the query tiles that see this key tile.
//   warps 0-7   compute: warp w owns TMEM lanes 32*(w%4).. (key rows) and query
//               columns 64*(w/4).. of each tile:
//                 P^T = exp2(S^T * scale*log2e - LSE*log2e)  -> TMEM (bf16, A of dV)
//                 dS^T = P^T (dP^T - Delta)                 -> smem (bf16, A of dK / dQ)
//               then drain dQ (lanes = query rows) into the fp32 accumulator
//               with vector atomics; finally the dV / dK epilogue.
//   warps 8-11  prologue (one warp per row at a time): K' once, then for every
//               query tile Q' = RoPE(RMSNorm(q)) into a 2-stage ring (bf16,
//               128B swizzle) plus the tile's LSE (base 2) and Delta.
//   warp 12     TMEM allocation + tcgen05.mma issue (one thread)
//   warp 13     TMA: V once, dO tiles into a 2-stage ring
// TMEM (512 columns): S^T/P^T/dQ | dP^T | dV | dK.
// MMA order per query tile n: [S(n) dP(n)] .. [dV(n) dK(n) dQ(n)] [dP(n+1)]
// [S(n+1) after dQ(n) is drained]; dQ(n) reuses the S columns once dV(n) has
// read P(n), so the drain overlaps dP(n+1).
#include "st_common.cuh"
#include "st_kernels.h"
#include "st_prologue.cuh"

namespace st {

namespace {

constexpr int kBwdWarps = 14;
constexpr int kBwdThreads = kBwdWarps * 32;
constexpr int kWarpProl0 = 8, kWarpMma = 12, kWarpTma = 13;
constexpr int kQStages = 2;

constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kTileBytes;
constexpr uint32_t kOffQ = 2 * kTileBytes;                    // kQStages tiles
constexpr uint32_t kOffDO = kOffQ + kQStages * kTileBytes;     // kQStages tiles
constexpr uint32_t kOffDS = kOffDO + kQStages * kTileBytes;
constexpr uint32_t kOffStat = kOffDS + kTileBytes;            // [stage][LSE*log2e | Delta][128] fp32
constexpr uint32_t kOffBar = kOffStat + kQStages * 2 * 128 * 4;
constexpr uint32_t kOffW = kOffBar + 256;                       // q norm weights, fp32
constexpr uint32_t kBwdSmem = kOffW + kD * 4;                   // the base must be 1024-byte aligned

enum {
  kBarKRaw = 0,                       // raw k rows landed (TMA)
  kBarKFull,
  kBarVFull,
  kBarQRaw,                           // + stage: raw q rows landed (TMA)
  kBarQFull = kBarQRaw + kQStages,    // + stage (prologue, 128 arrivals)
  kBarDOFull = kBarQFull + kQStages,  // + stage (TMA)
  kBarStageEmpty = kBarDOFull + kQStages,  // + stage (MMA commit)
  kBarSdPFull = kBarStageEmpty + kQStages,
  kBarPdSFull,                        // 256 arrivals
  kBarDQFull,
  kBarSFree,                          // 256 arrivals
  kBarFinal,                          // abort path: all issued MMAs done
  kNumBars
};

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, kHalfBytes, 1024);
}

__device__ __forceinline__ uint8_t tile_flag(const Common& c, int b, int h, int qt, int kt) {
  if (c.mask_kind == kMaskBool) return c.flags[b * c.f_sb + h * c.f_sh + qt * c.f_sq + kt];
  if (c.mask_kind == kMaskNone) return kTileAllTrue;
  return kTileMixed;
}

__device__ __forceinline__ int next_qtile(const Common& c, int b, int h, int qt, int kt) {
  if (c.mask_kind != kMaskBool) return qt;
  while (qt < c.nQt && tile_flag(c, b, h, qt, kt) == kTileAllFalse) ++qt;
  return qt;
}

__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(const __grid_constant__ BwdParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_u32(sm) & 1023u) {  // the layout has no slack: refuse an unaligned base
    if (threadIdx.x == 0) atomicOr(P.c.status, kStatusLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  float* stat = reinterpret_cast<float*>(sm + kOffStat);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const Common& c = P.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;

  if (warp == kWarpMma) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars[kBarKRaw], 1);
    mbar_init(&bars[kBarKFull], 128);
    mbar_init(&bars[kBarVFull], 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars[kBarQRaw + s], 1);
      mbar_init(&bars[kBarQFull + s], 128);
      mbar_init(&bars[kBarDOFull + s], 1);
      mbar_init(&bars[kBarStageEmpty + s], 1);
    }
    mbar_init(&bars[kBarSdPFull], 1);
    mbar_init(&bars[kBarPdSFull], 256);
    mbar_init(&bars[kBarDQFull], 1);
    mbar_init(&bars[kBarSFree], 256);
    mbar_init(&bars[kBarFinal], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  float* sWq = reinterpret_cast<float*>(sm + kOffW);
  if (tid < kD) sWq[tid] = __ldg(P.c.wq + tid);
  if (warp == kWarpTma && lane_id == 0) {
    tma_prefetch_desc(&P.tmap_v);
    tma_prefetch_desc(&P.tmap_do);
    if (P.qk_tma) {
      tma_prefetch_desc(&P.tmap_q);
      tma_prefetch_desc(&P.tmap_k);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const long long budget = c.wait_budget;
  const int qt_begin = c.causal ? min(c.nQt, (kt * kTile) / kTile) : 0;
  int processed = 0;  // query tiles processed (same count in every role)

  if (warp < 8) {
    // ------------------------------------------------------------ compute
    const int r = (warp & 3) * 32 + lane_id;  // key row in the tile / TMEM lane
    const int half = warp >> 2;               // query columns [64*half, 64*half + 64)
    const int j = kt * kTile + r;
    const bool key_ok = j < c.Skv;
    const uint32_t lane = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane, tdP = tmem + 128 + lane;
    // masks that do not depend on the query row: one term per key for the CTA
    float key_term = 0.f;
    const bool mask_bcast_q = c.mask_kind != kMaskNone && c.m_sq == 0;
    if (mask_bcast_q && key_ok) {
      const int64_t off = b * c.m_sb + h * c.m_sh + j;
      if (c.mask_kind == kMaskBool) key_term = __ldg(static_cast<const uint8_t*>(c.mask) + off) ? 0.f : -INFINITY;
      else if (c.mask_kind == kMaskF32) key_term = __ldg(static_cast<const float*>(c.mask) + off) * kLog2e;
      else key_term = __bfloat162float(static_cast<const __nv_bfloat16*>(c.mask)[off]) * kLog2e;
    }
    if (!key_ok) key_term = -INFINITY;
    bool ok = true;
    int n = 0;
    for (int qt = next_qtile(c, b, h, qt_begin, kt); qt < c.nQt; qt = next_qtile(c, b, h, qt + 1, kt), ++n) {
      const uint8_t flag = tile_flag(c, b, h, qt, kt);
      if (!(ok = wait_bar(&bars[kBarSdPFull], n & 1, abort_flag, budget))) break;
      tc_fence_after();
      // the prologue's LSE/Delta writes for this stage (already complete: the
      // MMA issue waited on the same phase) become visible through this wait
      if (!(ok = wait_bar(&bars[kBarQFull + n % kQStages], (n / kQStages) & 1, abort_flag, budget))) break;
      const float* st_lse = stat + (n % kQStages) * 256;
      const float* st_dl = st_lse + 128;
      uint32_t pw[32];  // P^T of this warp's 64 query columns, bf16 pairs
      // plain tiles: every query row valid, no mask values, no causal diagonal
      const bool plain = (qt + 1) * kTile <= c.Sq && (c.mask_kind == kMaskNone || mask_bcast_q ||
                                                      (c.mask_kind == kMaskBool && flag == kTileAllTrue)) &&
                         (!c.causal || kt < qt);
      const float sc = c.scale_log2;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int cbase = 64 * half + 16 * q4;  // first query column of this 16-column chunk
        uint32_t sv[16], dpv[16];
        tmem_ld16(tS + cbase, sv);
        tmem_ld16(tdP + cbase, dpv);
        float lse2[16], dl[16];
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const float4 a = *reinterpret_cast<const float4*>(st_lse + cbase + 4 * v4);
          const float4 d = *reinterpret_cast<const float4*>(st_dl + cbase + 4 * v4);
          lse2[4 * v4] = a.x; lse2[4 * v4 + 1] = a.y; lse2[4 * v4 + 2] = a.z; lse2[4 * v4 + 3] = a.w;
          dl[4 * v4] = d.x; dl[4 * v4 + 1] = d.y; dl[4 * v4 + 2] = d.z; dl[4 * v4 + 3] = d.w;
        }
        float pv[16], dsv[16];
        if (plain) {
#pragma unroll
          for (int t = 0; t < 16; ++t) pv[t] = ex2(fmaf(__uint_as_float(sv[t]), sc, key_term - lse2[t]));
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int iq = qt * kTile + cbase + t;
            float s2 = fmaf(__uint_as_float(sv[t]), sc, key_term);
            if (iq < c.Sq && !mask_bcast_q && c.mask_kind != kMaskNone && key_ok &&
                !(c.mask_kind == kMaskBool && flag == kTileAllTrue)) {
              const int64_t off = b * c.m_sb + h * c.m_sh + (int64_t)iq * c.m_sq + j;
              if (c.mask_kind == kMaskBool) {
                if (!__ldg(static_cast<const uint8_t*>(c.mask) + off)) s2 = -INFINITY;
              } else if (c.mask_kind == kMaskF32) {
                s2 = fmaf(__ldg(static_cast<const float*>(c.mask) + off), kLog2e, s2);
              } else {
                s2 = fmaf(__bfloat162float(static_cast<const __nv_bfloat16*>(c.mask)[off]), kLog2e, s2);
              }
            }
            if (c.causal && j > iq) s2 = -INFINITY;
            pv[t] = ex2(s2 - lse2[t]);  // lse2 = +inf for rows without keys or past S_q: P = 0
          }
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) dsv[t] = pv[t] * (__uint_as_float(dpv[t]) - dl[t]);
#pragma unroll
        for (int t = 0; t < 8; ++t) pw[8 * q4 + t] = pack_bf16(pv[2 * t], pv[2 * t + 1]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {  // dS^T row r, query columns cbase + 8u .. +7
          const int chunk = (cbase >> 3) + u;  // 16-byte chunk 0..15 along the query dimension
          *reinterpret_cast<uint4*>(sm + kOffDS + (chunk >> 3) * kHalfBytes + sw128_off(r, chunk & 7)) =
              make_uint4(pack_bf16(dsv[8 * u], dsv[8 * u + 1]), pack_bf16(dsv[8 * u + 2], dsv[8 * u + 3]),
                         pack_bf16(dsv[8 * u + 4], dsv[8 * u + 5]), pack_bf16(dsv[8 * u + 6], dsv[8 * u + 7]));
        }
      }
      // P^T overwrites S^T columns [32*half, 32*half + 32): wait until the other
      // warp on these lanes has read its S^T columns
      tc_fence_before();
      asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
      tc_fence_after();
      tmem_st32(tS + 32 * half, pw);
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kBarPdSFull]);
      // ---- dQ drain: lane = query row qt*128 + r, columns [64*half, +64). The
      // slice is read into registers and the S columns are released before the
      // reduction into the fp32 accumulator is issued, so the next S^T MMA does
      // not wait for the atomic traffic.
      if (!(ok = wait_bar(&bars[kBarDQFull], n & 1, abort_flag, budget))) break;
      tc_fence_after();
      uint32_t dq0[32], dq1[32];
      tmem_ld32(tS + 64 * half, dq0);
      tmem_ld32(tS + 64 * half + 32, dq1);
      tc_fence_before();
      mbar_arrive(&bars[kBarSFree]);
      const int iq = qt * kTile + r;
      if (iq < c.Sq) {
        float* dst = P.dq_acc + (((int64_t)b * c.Sq + iq) * c.H + h) * kD + 64 * half;
        const float sc2 = c.scale;
#pragma unroll
        for (int t = 0; t < 32; t += 4)
          red_add_v4(dst + t, __uint_as_float(dq0[t]) * sc2, __uint_as_float(dq0[t + 1]) * sc2,
                     __uint_as_float(dq0[t + 2]) * sc2, __uint_as_float(dq0[t + 3]) * sc2);
#pragma unroll
        for (int t = 0; t < 32; t += 4)
          red_add_v4(dst + 32 + t, __uint_as_float(dq1[t]) * sc2, __uint_as_float(dq1[t + 1]) * sc2,
                     __uint_as_float(dq1[t + 2]) * sc2, __uint_as_float(dq1[t + 3]) * sc2);
      }
    }
    processed = n;
    // ---- epilogue: warps 0-3 write dV, warps 4-7 dK (+ k-norm weight partials)
    if (ok) {
      tc_fence_after();
      float* red = reinterpret_cast<float*>(sm + kOffQ);  // [128][129] fp32 over the Q'/dO rings
      if (half == 0) {
        const int64_t off = b * P.dv_sb + (int64_t)j * P.dv_ss + h * P.dv_sh;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t v[32];
          if (n > 0) {
            tmem_ld32(tmem + 256 + lane + 32 * q4, v);
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = 0u;
          }
          float y[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) y[t] = __uint_as_float(v[t]);
          if (key_ok) store_chunk32(P.dv, off, P.dv_f32, q4, y);
        }
      } else {
        // dK' (TMEM, 32 columns at a time) -> inverse rotation -> RMSNorm backward.
        //   dy = R^T (scale dK'), g = w dy, dx = r g - (r^3 / D) x (x . g);
        // the weight-gradient term dy x r goes to the shared reduction buffer.
        float* my = red + r * (kD + 1);
        const int64_t xoff = b * c.k.sb + (int64_t)j * c.k.ss + h * c.k.sh;
        const float2* tab = c.tab_k + b * c.tab_k_sb + (int64_t)j * kPairs;
        float rr = 0.f;
        if (key_ok) {
          float ss0 = 0.f, ss1 = 0.f;
#pragma unroll 4
          for (int cc = 0; cc < kD / 8; ++cc) {
            float x[8];
            load_chunk8(c.k.p, xoff, c.k.is_f32, cc, x);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              ss0 = fmaf(x[e], x[e], ss0);
              ss1 = fmaf(x[e + 1], x[e + 1], ss1);
            }
          }
          rr = rsqrtf((ss0 + ss1) * (1.0f / kD) + c.eps);
        }
        float xg = 0.f;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          const float c3 = rr * rr * rr * xg * (1.0f / kD);
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t v[32];
            if (n > 0) {
              tmem_ld32(tmem + 384 + lane + 32 * q4, v);
            } else {
#pragma unroll
              for (int t = 0; t < 32; ++t) v[t] = 0u;
            }
            if (!key_ok) continue;
            float y[32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              float x[8];
              load_chunk8(c.k.p, xoff, c.k.is_f32, 4 * q4 + cc, x);
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const int t = 8 * cc + e, d = 32 * q4 + t;
                const float2 cs = __ldg(tab + d / 2);
                const float g0 = __uint_as_float(v[t]) * c.scale, g1 = __uint_as_float(v[t + 1]) * c.scale;
                const float d0 = g0 * cs.x + g1 * cs.y;    // inverse rotation (sin negated)
                const float d1 = -g0 * cs.y + g1 * cs.x;
                const float w0 = __ldg(c.wk + d), w1 = __ldg(c.wk + d + 1);
                if (pass == 0) {
                  my[d] = d0 * (x[e] * rr);
                  my[d + 1] = d1 * (x[e + 1] * rr);
                  xg = fmaf(x[e], w0 * d0, fmaf(x[e + 1], w1 * d1, xg));
                } else {
                  y[t] = rr * (w0 * d0) - c3 * x[e];
                  y[t + 1] = rr * (w1 * d1) - c3 * x[e + 1];
                }
              }
            }
            if (pass == 1) store_chunk32(P.dk, b * P.dk_sb + (int64_t)j * P.dk_ss + h * P.dk_sh, P.dk_f32, q4, y);
          }
        }
        if (!key_ok) {
          for (int d = 0; d < kD; ++d) my[d] = 0.f;
        }
      }
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ prologue
    const int p = tid - kWarpProl0 * 32;  // row of the tile handled by this thread
    bool ok = true;
    {
      const int j = kt * kTile + p;
      const float2* tab = c.tab_k + b * c.tab_k_sb + (int64_t)j * kPairs;
      if (P.qk_tma) {
        ok = wait_bar(&bars[kBarKRaw], 0, abort_flag, budget);
        if (ok && j < c.Skv)  // rows past S_kv stay zero
          rope_norm_inplace(sm + kOffK, p, c.wk, c.eps, c.tab16_k + b * c.tab_k_sb + (int64_t)j * kPairs);
      } else if (j < c.Skv) {
        rope_norm_global(c.k.p, b * c.k.sb + (int64_t)j * c.k.ss + h * c.k.sh, c.k.is_f32, c.wk, c.eps, tab,
                         sm + kOffK, p);
      } else {
        zero_row(sm + kOffK, p);
      }
      if (ok) {
        fence_proxy_async_smem();
        mbar_arrive(&bars[kBarKFull]);
      }
    }
    int n = 0;
    for (int qt = next_qtile(c, b, h, qt_begin, kt); ok && qt < c.nQt; qt = next_qtile(c, b, h, qt + 1, kt), ++n) {
      const int s = n % kQStages;
      uint8_t* tile = sm + kOffQ + s * kTileBytes;
      const int i = qt * kTile + p;
      const float2* tab = c.tab_q + b * c.tab_q_sb + (int64_t)i * kPairs;
      if (P.qk_tma) {
        if (!wait_bar(&bars[kBarQRaw + s], (n / kQStages) & 1, abort_flag, budget)) break;
        if (i < c.Sq) rope_norm_inplace(tile, p, sWq, c.eps, c.tab16_q + b * c.tab_q_sb + (int64_t)i * kPairs);
      } else {
        if (n >= kQStages && !wait_bar(&bars[kBarStageEmpty + s], ((n / kQStages) - 1) & 1, abort_flag, budget))
          break;
        if (i < c.Sq)
          rope_norm_global(c.q.p, b * c.q.sb + (int64_t)i * c.q.ss + h * c.q.sh, c.q.is_f32, c.wq, c.eps, tab, tile,
                           p);
        else
          zero_row(tile, p);
      }
      {  // this tile's LSE (base 2; +inf for rows without keys, so P = 0) and Delta
        float l2 = INFINITY, dl = 0.f;
        if (i < c.Sq) {
          const int64_t rr = ((int64_t)b * c.H + h) * c.Sq + i;
          const float l = __ldg(P.lse + rr);
          l2 = (l == -INFINITY) ? INFINITY : l * kLog2e;
          dl = __ldg(P.delta + rr);
        }
        stat[s * 256 + p] = l2;
        stat[s * 256 + 128 + p] = dl;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[kBarQFull + s]);
    }
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA: raw K, V, raw Q, dO
    if (lane_id == 0) {
      if (P.qk_tma) {
        const int y = P.k_s_first ? kt * kTile : h, z = P.k_s_first ? h : kt * kTile;
        mbar_arrive_expect_tx(&bars[kBarKRaw], kTileBytes);
        tma_load_4d(sm + kOffK, &P.tmap_k, &bars[kBarKRaw], 0, y, z, b);
        tma_load_4d(sm + kOffK + kHalfBytes, &P.tmap_k, &bars[kBarKRaw], 64, y, z, b);
      }
      const int vy = P.v_s_first ? kt * kTile : h, vz = P.v_s_first ? h : kt * kTile;
      mbar_arrive_expect_tx(&bars[kBarVFull], kTileBytes);
      tma_load_4d(sm + kOffV, &P.tmap_v, &bars[kBarVFull], 0, vy, vz, b);
      tma_load_4d(sm + kOffV + kHalfBytes, &P.tmap_v, &bars[kBarVFull], 64, vy, vz, b);
      int n = 0;
      for (int qt = next_qtile(c, b, h, qt_begin, kt); qt < c.nQt; qt = next_qtile(c, b, h, qt + 1, kt), ++n) {
        const int s = n % kQStages;
        if (n >= kQStages && !wait_bar(&bars[kBarStageEmpty + s], ((n / kQStages) - 1) & 1, abort_flag, budget))
          break;
        if (P.qk_tma) {
          uint8_t* qtile = sm + kOffQ + s * kTileBytes;
          const int y = P.q_s_first ? qt * kTile : h, z = P.q_s_first ? h : qt * kTile;
          mbar_arrive_expect_tx(&bars[kBarQRaw + s], kTileBytes);
          tma_load_4d(qtile, &P.tmap_q, &bars[kBarQRaw + s], 0, y, z, b);
          tma_load_4d(qtile + kHalfBytes, &P.tmap_q, &bars[kBarQRaw + s], 64, y, z, b);
        }
        uint8_t* tile = sm + kOffDO + s * kTileBytes;
        const int y = P.do_s_first ? qt * kTile : h, z = P.do_s_first ? h : qt * kTile;
        mbar_arrive_expect_tx(&bars[kBarDOFull + s], kTileBytes);
        tma_load_4d(tile, &P.tmap_do, &bars[kBarDOFull + s], 0, y, z, b);
        tma_load_4d(tile + kHalfBytes, &P.tmap_do, &bars[kBarDOFull + s], 64, y, z, b);
      }
      // drain: every issued load lands before the CTA exits
      wait_bar(&bars[kBarVFull], 0, abort_flag, budget);
      if (P.qk_tma) wait_bar(&bars[kBarKRaw], 0, abort_flag, budget);
      for (int m = max(0, n - kQStages); m < n; ++m) {
        wait_bar(&bars[kBarDOFull + m % kQStages], (m / kQStages) & 1, abort_flag, budget);
        if (P.qk_tma) wait_bar(&bars[kBarQRaw + m % kQStages], (m / kQStages) & 1, abort_flag, budget);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue
    if (lane_id == 0) {
      const uint32_t idesc_kk = idesc_bf16(128, 128, 0, 0);
      const uint32_t idesc_kmn = idesc_bf16(128, 128, 0, 1);
      const uint32_t idesc_mnmn = idesc_bf16(128, 128, 1, 1);
      const uint32_t aK = smem_u32(sm + kOffK), aV = smem_u32(sm + kOffV), adS = smem_u32(sm + kOffDS);
      const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
      bool ok = wait_bar(&bars[kBarKFull], 0, abort_flag, budget) && wait_bar(&bars[kBarVFull], 0, abort_flag, budget);
      int qt = next_qtile(c, b, h, qt_begin, kt);
      int n = 0;
      bool issued = false;
      if (ok && qt < c.nQt) {
        ok = wait_bar(&bars[kBarQFull], 0, abort_flag, budget) && wait_bar(&bars[kBarDOFull], 0, abort_flag, budget);
        if (ok) {
          tc_fence_after();
          const uint32_t aQ = smem_u32(sm + kOffQ), adO = smem_u32(sm + kOffDO);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tdP, kmajor_desc(aV, kk), kmajor_desc(adO, kk), idesc_kk, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS, kmajor_desc(aK, kk), kmajor_desc(aQ, kk), idesc_kk, kk > 0);
          mma_commit(&bars[kBarSdPFull]);
          issued = true;
        }
      }
      while (ok && qt < c.nQt) {
        const int s = n % kQStages;
        const uint32_t aQ = smem_u32(sm + kOffQ + s * kTileBytes), adO = smem_u32(sm + kOffDO + s * kTileBytes);
        if (!(ok = wait_bar(&bars[kBarPdSFull], n & 1, abort_flag, budget))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts(tdV, tS + kk * 8, mnmajor_desc(adO, kk), idesc_kmn, (n > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tdK, kmajor_desc(adS, kk), mnmajor_desc(aQ, kk), idesc_kmn, (n > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tS, mnmajor_desc(adS, kk), mnmajor_desc(aK, kk), idesc_mnmn, kk > 0);
        mma_commit(&bars[kBarDQFull]);
        mma_commit(&bars[kBarStageEmpty + s]);
        const int qt_next = next_qtile(c, b, h, qt + 1, kt);
        if (qt_next < c.nQt) {
          const int ns = (n + 1) % kQStages, nph = ((n + 1) / kQStages) & 1;
          if (!(ok = wait_bar(&bars[kBarQFull + ns], nph, abort_flag, budget))) break;
          if (!(ok = wait_bar(&bars[kBarDOFull + ns], nph, abort_flag, budget))) break;
          tc_fence_after();
          const uint32_t aQn = smem_u32(sm + kOffQ + ns * kTileBytes), adOn = smem_u32(sm + kOffDO + ns * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tdP, kmajor_desc(aV, kk), kmajor_desc(adOn, kk), idesc_kk, kk > 0);
          if (!(ok = wait_bar(&bars[kBarSFree], n & 1, abort_flag, budget))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tS, kmajor_desc(aK, kk), kmajor_desc(aQn, kk), idesc_kk, kk > 0);
          mma_commit(&bars[kBarSdPFull]);
        }
        qt = qt_next;
        ++n;
      }
      if (issued && !ok) {
        // abort: let every issued MMA finish before TMEM is released
        mma_commit(&bars[kBarFinal]);
        const long long t0 = clock64();
        while (!mbar_try_wait(&bars[kBarFinal], 0) && clock64() - t0 < budget) {
        }
      }
    }
  }

  // ---- k-norm weight partials: column sums of the dK warps' contributions
  tc_fence_before();
  __syncthreads();
  if (!*abort_flag) {
    if (tid < kD) {
      const float* red = reinterpret_cast<const float*>(sm + kOffQ);
      float acc = 0.f;
      for (int r = 0; r < kTile; ++r) acc += red[r * (kD + 1) + tid];
      P.dwk_part[(((int64_t)b * c.H + h) * c.nKt + kt) * kD + tid] = acc;
    }
    if (tid == 0) {
      const int total = c.nQt - qt_begin;
      atomicAdd(c.counters + kCtrTilesSkipped, (unsigned long long)(c.nQt - processed));
      atomicAdd(c.counters + kCtrTilesTotal, (unsigned long long)c.nQt);
      (void)total;
    }
  } else if (tid == 0) {
    record_timeout(c);
  }
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
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
