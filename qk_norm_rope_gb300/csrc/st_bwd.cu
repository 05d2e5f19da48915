// Backward main kernel: one CTA per (key tile of 128 rows, head, batch), in
// clusters of two CTAs over adjacent key tiles (kt0 = 2p, kt0 + 1) that walk
// the same query tiles in lockstep. Per query tile, with Q' = RoPE(RMSNorm(q))
// and K' the same for k (bf16, 128B-swizzled operand tiles):
//   S^T = K' Q'^T, dP^T = V dO^T                      (tensor core, TMEM)
//   P^T = exp2(S^T scale log2e - LSE log2e)            (compute warps)
//   dS^T = P^T (dP^T - Delta)
//   dV += P^T dO, dK += dS^T Q', dQ_part = dS K'       (tensor core, TMEM)
// dQ_part (this CTA's 128 keys) is added into a global fp32 accumulator by TMA
// bulk reduces. The two CTAs of a cluster share the Q' operand prologue.
//
// Warp roles (576 threads; 96 registers per thread):
//   warps 0-7    compute: warp w owns TMEM lanes 32*(w%4).. (key rows) and
//                query columns [64*(w/4), +64) of each tile; P^T goes to TMEM
//                (bf16, in the warp's own S^T columns: 0-31 for the first query
//                half, 96-127 for the second), dS^T to shared memory
//   warps 8-11   dQ drain: TMEM lanes = query rows; B is read out at once
//                (half staged in shared memory, half held in registers) and
//                released, then reduced to global memory by TMA in two rounds
//   warps 12-15  Q' prologue: each CTA of the cluster normalises and rotates
//                64 of the tile's 128 rows (eight lanes per row) and copies them
//                into the peer's stage as well (DSMEM bulk copy); the tile's
//                LSE and Delta; K' once
//   warp 16      TMEM allocation + tcgen05.mma issue (one thread)
//   warp 17      TMA: raw K, V once; this CTA's 64 raw Q rows per tile (2-stage
//                ring, a stage reused once both CTAs' MMAs released it); dO in
//                two 64-row halves, each refilled as soon as its dV MMAs ran
// TMEM (512 columns): A = S^T / P^T | B = dP^T / dQ | dV | dK.
// MMA order per query tile n:
//   [half 0 done] dV, dK over queries 0-63 | [half 1 done] dV, dK over
//   queries 64-127, dQ (into B) | S^T(n+1) (into A) | [B drained] dP^T(n+1)
// so the tensor core computes the next tile's scores while the drain warps
// empty B.
#include "st_common.cuh"
#include "st_kernels.h"
#include "st_prologue.cuh"

namespace st {

namespace {

constexpr int kCluster = 2;
constexpr int kComputeWarps = 8;
constexpr int kWarpDrain0 = 8, kDrainWarps = 4;
constexpr int kWarpProl0 = 12, kProlWarps = 4;
constexpr int kWarpMma = 16, kWarpTma = 17;
constexpr int kBwdWarps = 18;
constexpr int kProlThreads = kProlWarps * 32;
constexpr int kBwdThreads = kBwdWarps * 32;
constexpr int kQStages = 2;
constexpr uint32_t kRBoxBytes = kTile * 32 * 4;  // one [128 query rows][32 head dims] fp32 box, 128B-swizzled
constexpr int kHalfRows = kTile / kCluster;                      // Q' rows produced per CTA
constexpr uint32_t kHalfRowsBytes = kHalfRows * 128;             // those rows in one 64-column half

// shared memory layout (offsets from the 1024-byte aligned dynamic base)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kTileBytes;
constexpr uint32_t kOffQ = 2 * kTileBytes;                  // kQStages tiles
constexpr uint32_t kOffDO = kOffQ + kQStages * kTileBytes;  // rows 0-63 / 64-127 refilled separately
constexpr uint32_t kOffDS = kOffDO + kTileBytes;
constexpr uint32_t kOffR = kOffDS + kTileBytes;             // dQ staging: 2 boxes of 32 head dims
constexpr uint32_t kOffStat = kOffR + 2 * kRBoxBytes;       // [stage][LSE*log2e | Delta][128] fp32
constexpr uint32_t kOffBar = kOffStat + kQStages * 2 * kTile * 4;
constexpr uint32_t kOffW = kOffBar + 256;                   // q norm weights, fp32
constexpr uint32_t kBwdSmem = kOffW + kD * 4;               // the base must be 1024-byte aligned
static_assert(kBwdSmem <= 232448, "backward shared memory exceeds the per-block limit");

enum {
  kBarKRaw = 0,                          // raw k rows landed (TMA)
  kBarKFull,                             // K' ready (and V, for a CTA past the last key tile)
  kBarVFull,
  kBarQRaw,                              // + stage: raw q rows landed (TMA)
  kBarQFull = kBarQRaw + kQStages,       // + stage: Q' + stats ready (prologue threads + the peer's rows)
  kBarQFree = kBarQFull + kQStages,      // + stage: both CTAs' MMAs done with the stage
  kBarDOLoFull = kBarQFree + kQStages,   // dO rows 0-63 landed
  kBarDOHiFull,                          // dO rows 64-127 landed
  kBarDOLoFree,                          // MMAs done with dO rows 0-63
  kBarDOHiFree,
  kBarSFull,                             // S^T in A
  kBarDPFull,                            // dP^T in B
  kBarHalf0,                             // compute warps of query half 0 done (128 arrivals)
  kBarHalf1,
  kBarDQFull,                            // dQ partial in B (and every earlier MMA done)
  kBarBFree,                             // B drained (128 arrivals)
  kBarFinal,                             // abort path: all issued MMAs done
  kNumBars
};
static_assert(kNumBars * 8 + 12 <= 256, "barrier area");
static_assert(kTile % kProlThreads == 0 && kProlThreads <= kTile, "prologue threads cover the stat rows evenly");

__device__ __forceinline__ uint32_t kofs(int kk) { return (kk >> 2) * kHalfBytes + (kk & 3) * 32; }  // K-major step
__device__ __forceinline__ uint32_t mofs(int kk) { return kk * 2048; }                               // MN-major step

// Tile class of (query tile qt, key tile kt) for this CTA's own key tile; a
// CTA past the last key tile sees nothing.
template <int MK>
__device__ __forceinline__ uint8_t own_flag(const Common& c, int b, int h, int qt, int kt) {
  if (kt >= c.nKt) return kTileAllFalse;
  if constexpr (MK == kMaskBool) return c.flags[b * c.f_sb + h * c.f_sh + qt * c.f_sq + kt];
  if constexpr (MK == kMaskNone) return kTileAllTrue;
  return kTileMixed;
}

// The query tiles a cluster visits: [begin, begin + len), walked from a
// rotated start so that the clusters of one head (which all add into the same
// dQ rows) do not work on the same query tile at the same time.
struct QWalk {
  int begin, len, rot;
  __device__ __forceinline__ int qt(int m) const {
    const int x = rot + m;
    return begin + (x >= len ? x - len : x);
  }
};

// Next walk position at or after m whose query tile either key tile of the
// cluster needs.
template <int MK>
__device__ __forceinline__ int next_pos(const Common& c, int b, int h, const QWalk& w, int m, int kt0) {
  if constexpr (MK == kMaskBool) {
    while (m < w.len && own_flag<MK>(c, b, h, w.qt(m), kt0) == kTileAllFalse &&
           own_flag<MK>(c, b, h, w.qt(m), kt0 + 1) == kTileAllFalse)
      ++m;
  }
  return m;
}

// Base-2 score of key j against query iq (general path): s*scale*log2e plus
// the key's broadcast term, the per-element mask, causal and bounds.
template <int MK, bool CAUSAL>
__device__ __forceinline__ float score2(const Common& c, float s, float key_term, int b, int h, int iq, int j,
                                        bool key_ok, uint8_t flag, bool mask_bcast_q) {
  float s2 = fmaf(s, c.scale_log2, key_term);
  if (flag == kTileAllFalse) return -INFINITY;
  if constexpr (MK != kMaskNone) {
    if (!mask_bcast_q && key_ok && iq < c.Sq && !(MK == kMaskBool && flag == kTileAllTrue)) {
      const int64_t off = b * c.m_sb + h * c.m_sh + (int64_t)iq * c.m_sq + j;
      if constexpr (MK == kMaskBool) {
        if (!__ldg(static_cast<const uint8_t*>(c.mask) + off)) s2 = -INFINITY;
      } else if constexpr (MK == kMaskF32) {
        s2 = fmaf(__ldg(static_cast<const float*>(c.mask) + off), kLog2e, s2);
      } else {
        s2 = fmaf(__bfloat162float(static_cast<const __nv_bfloat16*>(c.mask)[off]), kLog2e, s2);
      }
    }
  }
  if constexpr (CAUSAL) {
    if (j > iq) s2 = -INFINITY;
  }
  return s2;
}

// As score2, with the element's mask term already loaded (mterm: mask*log2e,
// -inf for a False bool element, 0 where no mask applies).
template <bool CAUSAL>
__device__ __forceinline__ float score2_term(const Common& c, float s, float key_term, float mterm, int iq, int j,
                                             uint8_t flag) {
  if (flag == kTileAllFalse) return -INFINITY;
  float s2 = fmaf(s, c.scale_log2, key_term) + mterm;
  if constexpr (CAUSAL) {
    if (j > iq) s2 = -INFINITY;
  }
  return s2;
}

// ELEM: the mask varies along the queries (per-element terms); a mask that is
// broadcast over the queries reduces to one term per key.
template <int MK, bool CAUSAL, bool QKT, bool ELEM>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ BwdParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_u32(sm) & 1023u) {  // the layout has no slack: refuse an unaligned base (uniform over the grid)
    if (threadIdx.x == 0) atomicOr(P.c.status, kStatusLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  float* stat = reinterpret_cast<float*>(sm + kOffStat);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  uint32_t* scratch = tslot + 2;  // sink for pin_loads

  const Common& c = P.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int kt0 = kt & ~1;

  if (warp == kWarpMma) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars[kBarKRaw], 1);
    mbar_init(&bars[kBarKFull], kProlThreads);
    mbar_init(&bars[kBarVFull], 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars[kBarQRaw + s], 1);
      mbar_init(&bars[kBarQFull + s], kProlThreads);
      mbar_init(&bars[kBarQFree + s], kCluster);
    }
    mbar_init(&bars[kBarDOLoFull], 1);
    mbar_init(&bars[kBarDOHiFull], 1);
    mbar_init(&bars[kBarDOLoFree], 1);
    mbar_init(&bars[kBarDOHiFree], 1);
    mbar_init(&bars[kBarSFull], 1);
    mbar_init(&bars[kBarDPFull], 1);
    mbar_init(&bars[kBarHalf0], 128);
    mbar_init(&bars[kBarHalf1], 128);
    mbar_init(&bars[kBarDQFull], 1);
    mbar_init(&bars[kBarBFree], kDrainWarps * 32);
    mbar_init(&bars[kBarFinal], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  float* sWq = reinterpret_cast<float*>(sm + kOffW);
  if (tid < kD) sWq[tid] = __ldg(P.c.wq + tid);
  if (warp == kWarpTma && lane_id == 0 && P.c.nQt > 0) {  // the maps exist only when there is work
    tma_prefetch_desc(&P.tmap_v);
    tma_prefetch_desc(&P.tmap_do);
    tma_prefetch_desc(&P.tmap_dq);
    if constexpr (QKT) {
      tma_prefetch_desc(&P.tmap_q);
      tma_prefetch_desc(&P.tmap_k);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote store or arrival
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t crank = cluster_rank(), peer = crank ^ 1u;
  const long long budget = c.wait_budget;
  const bool phantom = kt >= c.nKt;  // pads the cluster when the key-tile count is odd
  QWalk W;
  W.begin = CAUSAL ? min(c.nQt, kt0) : 0;
  W.len = c.nQt - W.begin;
  W.rot = W.len > 0 ? static_cast<int>((static_cast<int64_t>(kt0 / 2) * W.len) / ((c.nKt + 1) / 2)) : 0;
  int useful = 0;  // query tiles this CTA's own key tile needed (compute warps)

  if (warp < kComputeWarps) {
    // ------------------------------------------------------------ compute
    const int qd = warp & 3, hq = warp >> 2;  // TMEM lane quarter, query half
    const int r = qd * 32 + lane_id;          // key row in the tile / TMEM lane
    const int j = kt * kTile + r;
    const bool key_ok = j < c.Skv;
    const uint32_t lanebits = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t tA = tmem + lanebits, tB = tmem + 128 + lanebits;
    const uint32_t tP = tA + (hq ? 96 : 0);  // P^T of the warp's 64 queries, inside its own S^T columns
    // masks that do not depend on the query row: one term per key for the CTA
    float key_term = 0.f;
    const bool mask_bcast_q = MK != kMaskNone && c.m_sq == 0;
    if (mask_bcast_q && key_ok) {
      const int64_t off = b * c.m_sb + h * c.m_sh + j;
      if constexpr (MK == kMaskBool) key_term = __ldg(static_cast<const uint8_t*>(c.mask) + off) ? 0.f : -INFINITY;
      else if constexpr (MK == kMaskF32) key_term = __ldg(static_cast<const float*>(c.mask) + off) * kLog2e;
      else if constexpr (MK == kMaskBF16) key_term = __bfloat162float(static_cast<const __nv_bfloat16*>(c.mask)[off]) * kLog2e;
    }
    if (!key_ok) key_term = -INFINITY;
    const float sc = c.scale_log2;
    bool ok = true;
    int n = 0;
    for (int m = next_pos<MK>(c, b, h, W, 0, kt0); m < W.len; m = next_pos<MK>(c, b, h, W, m + 1, kt0), ++n) {
      const int qt = W.qt(m);
      const uint8_t flag = own_flag<MK>(c, b, h, qt, kt);
      useful += (flag != kTileAllFalse && (!CAUSAL || qt >= kt)) ? 1 : 0;
      const int s = n % kQStages;
      if (!(ok = wait_bar_warp(&bars[kBarSFull], n & 1, abort_flag, budget))) break;
      // the prologue's LSE/Delta for this stage become visible through this wait
      if (!(ok = wait_bar_warp(&bars[kBarQFull + s], (n / kQStages) & 1, abort_flag, budget))) break;
      tc_fence_after();
      const float* st_lse = stat + s * 256;
      const float* st_dl = st_lse + 128;
      // plain tiles: every query row valid, no mask values, no causal diagonal
      const bool plain = flag != kTileAllFalse && (qt + 1) * kTile <= c.Sq &&
                         (MK == kMaskNone || mask_bcast_q || (MK == kMaskBool && flag == kTileAllTrue)) &&
                         (!CAUSAL || kt < qt);
      // ---- P^T = exp2(S^T * scale*log2e - LSE*log2e), bf16 into TMEM. The
      // general path (masks, causal diagonal, ragged tiles) is kept apart so
      // that the plain loop stays short and contiguous in the instruction cache.
      uint32_t pw[32];
      if (plain) {
        const float2 sc2 = make_float2(sc, sc), kt2 = make_float2(key_term, key_term);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int q0 = 64 * hq + 32 * cc;  // first query column (in the tile) of this chunk
          uint32_t sv[32];
          tmem_ld32(tA + q0, sv);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const float4 l = *reinterpret_cast<const float4*>(st_lse + q0 + 4 * v4);
            const float2 c01 = __fadd2_rn(kt2, make_float2(-l.x, -l.y)), c23 = __fadd2_rn(kt2, make_float2(-l.z, -l.w));
            const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sv[4 * v4]), __uint_as_float(sv[4 * v4 + 1])), sc2, c01);
            const float2 x23 =
                __ffma2_rn(make_float2(__uint_as_float(sv[4 * v4 + 2]), __uint_as_float(sv[4 * v4 + 3])), sc2, c23);
            pw[16 * cc + 2 * v4] = pack_bf16(ex2(x01.x), ex2(x01.y));
            pw[16 * cc + 2 * v4 + 1] = pack_bf16(ex2(x23.x), ex2(x23.y));
          }
        }
      } else if constexpr (!ELEM) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int q0 = 64 * hq + 32 * cc;
          uint32_t sv[32];
          tmem_ld32(tA + q0, sv);
#pragma unroll
          for (int t2 = 0; t2 < 16; ++t2) {
            float p2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = 2 * t2 + e;
              const float s2 = score2<MK, CAUSAL>(c, __uint_as_float(sv[t]), key_term, b, h, qt * kTile + q0 + t, j,
                                                  key_ok, flag, mask_bcast_q);
              p2[e] = ex2(s2 - st_lse[q0 + t]);  // LSE = +inf for rows without keys or past S_q: P = 0
            }
            pw[16 * cc + t2] = pack_bf16(p2[0], p2[1]);
          }
        }
      } else {
        // 16 queries at a time; the next chunk's mask terms are loaded while
        // this one is computed (pinned at the end of the chunk)
        const bool elem_mask = ELEM && key_ok && flag != kTileAllFalse && !(MK == kMaskBool && flag == kTileAllTrue);
        float mv[2][16];
        uint32_t mraw[2][16];
        auto issue = [&](int c4, uint32_t (&raw)[16]) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            raw[t] = 0u;
            if constexpr (ELEM) {
              const int iq = qt * kTile + 64 * hq + 16 * c4 + t;
              if (elem_mask && iq < c.Sq) {
                const int64_t off = b * c.m_sb + h * c.m_sh + (int64_t)iq * c.m_sq + j;
                if constexpr (MK == kMaskBool) raw[t] = __ldg(static_cast<const uint8_t*>(c.mask) + off) ? 0u : 1u;
                else if constexpr (MK == kMaskF32)
                  raw[t] = __float_as_uint(ldg_nc_f32(static_cast<const float*>(c.mask) + off));
                else raw[t] = static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(c.mask) + off)) << 16;
              }
            }
          }
        };
        auto settle = [&](const uint32_t (&raw)[16], float (&m)[16]) {  // pin, then convert
          uint32_t folded = 0;
#pragma unroll
          for (int t = 0; t < 16; ++t) folded ^= raw[t];
          pin_loads(folded, scratch);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            if constexpr (MK == kMaskBool) m[t] = raw[t] ? -INFINITY : 0.f;
            else m[t] = __uint_as_float(raw[t]) * kLog2e;
          }
        };
        issue(0, mraw[0]);
        settle(mraw[0], mv[0]);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          if (c4 < 3) issue(c4 + 1, mraw[(c4 + 1) & 1]);
          const int q0 = 64 * hq + 16 * c4;  // first query column (in the tile) of this chunk
          uint32_t sv[16];
          tmem_ld16(tA + q0, sv);
#pragma unroll
          for (int t2 = 0; t2 < 8; ++t2) {
            float p2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = 2 * t2 + e;
              const float s2 = score2_term<CAUSAL>(c, __uint_as_float(sv[t]), key_term, mv[c4 & 1][t], qt * kTile + q0 + t, j, flag);
              p2[e] = ex2(s2 - st_lse[q0 + t]);  // LSE = +inf for rows without keys or past S_q: P = 0
            }
            pw[8 * c4 + t2] = pack_bf16(p2[0], p2[1]);
          }
          if (c4 < 3) settle(mraw[(c4 + 1) & 1], mv[(c4 + 1) & 1]);
        }
      }
      tmem_st32(tP, pw);
      // ---- dS^T = P^T (dP^T - Delta), bf16 into shared memory (row r, K-major)
      if (!(ok = wait_bar_warp(&bars[kBarDPFull], n & 1, abort_flag, budget))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int q0 = 64 * hq + 32 * cc;
        uint32_t dpv[32];
        tmem_ld32(tB + q0, dpv);
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // 8 queries = one 16-byte chunk of the dS^T row
          const float4 d0 = *reinterpret_cast<const float4*>(st_dl + q0 + 8 * u);
          const float4 d1 = *reinterpret_cast<const float4*>(st_dl + q0 + 8 * u + 4);
          const float2 ndl[4] = {make_float2(-d0.x, -d0.y), make_float2(-d0.z, -d0.w), make_float2(-d1.x, -d1.y),
                                 make_float2(-d1.z, -d1.w)};
          uint32_t out[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t pp = pw[16 * cc + 4 * u + e];
            const float2 dp = make_float2(__uint_as_float(dpv[8 * u + 2 * e]), __uint_as_float(dpv[8 * u + 2 * e + 1]));
            const float2 ds = __fmul2_rn(make_float2(bf16_lo(pp), bf16_hi(pp)), __fadd2_rn(dp, ndl[e]));
            out[e] = pack_bf16(ds.x, ds.y);
          }
          *reinterpret_cast<uint4*>(sm + kOffDS + hq * kHalfBytes + sw128_off(r, 4 * cc + u)) =
              make_uint4(out[0], out[1], out[2], out[3]);
        }
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kBarHalf0 + hq]);
    }
    // ---- epilogue: warps of query half 0 write dV, half 1 scale * dK' (fp32;
    // the inverse rotation and the RMSNorm backward run in a row kernel after)
    if (ok && n > 0) ok = wait_bar_warp(&bars[kBarDQFull], (n - 1) & 1, abort_flag, budget);
    if (ok) {
      tc_fence_after();
      const uint32_t tacc = tmem + (hq == 0 ? 256 : 384) + lanebits;
      const int64_t off = hq == 0 ? b * P.dv_sb + (int64_t)j * P.dv_ss + h * P.dv_sh
                                  : (((int64_t)b * c.Skv + j) * c.H + h) * kD;
      const float mul = hq == 0 ? 1.f : c.scale;
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(tacc + 32 * q4, v);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) v[t] = 0u;
        }
        float y[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) y[t] = __uint_as_float(v[t]) * mul;
        if (key_ok) {
          if (hq == 0) store_chunk32(P.dv, off, P.dv_f32, q4, y);
          else store_chunk32(P.dk_acc, off, 1, q4, y);
        }
      }
    }
  } else if (warp < kWarpDrain0 + kDrainWarps) {
    // ------------------------------------------------------------ dQ drain
    // The tile's partial dQ (128 query rows x 128 head dims, fp32) leaves B
    // at once: columns 0-63 are staged in shared memory, 64-127 held in
    // registers, then B is released; each half goes out as two TMA bulk
    // reduces (fp32 add into the global accumulator).
    const int qd = warp & 3;
    const int qrow = qd * 32 + lane_id;  // query row in the tile = TMEM lane
    const uint32_t tB = tmem + 128 + (static_cast<uint32_t>(qd * 32) << 16);
    uint8_t* R = sm + kOffR;
    const float scale = c.scale;
    const bool issuer = warp == kWarpDrain0 && lane_id == 0;
    auto stage32 = [&](int box, const uint32_t (&v)[32]) {  // 32 columns of this row into staging box `box`
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(R + box * kRBoxBytes + sw128_off(qrow, k)) =
            make_uint4(__float_as_uint(__uint_as_float(v[4 * k]) * scale),
                       __float_as_uint(__uint_as_float(v[4 * k + 1]) * scale),
                       __float_as_uint(__uint_as_float(v[4 * k + 2]) * scale),
                       __float_as_uint(__uint_as_float(v[4 * k + 3]) * scale));
    };
    int n = 0;
    for (int m = next_pos<MK>(c, b, h, W, 0, kt0); m < W.len; m = next_pos<MK>(c, b, h, W, m + 1, kt0), ++n) {
      const int qt = W.qt(m);
      // A failed wait skips the work but not the named barriers below; every
      // thread then leaves together on the abort flag.
      const bool ok = wait_bar_warp(&bars[kBarDQFull], n & 1, abort_flag, budget);
      uint32_t hold0[32], hold1[32];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t v[32];
          tmem_ld32(tB + 32 * cc, v);
          stage32(cc, v);
        }
        tmem_ld32(tB + 64, hold0);
        tmem_ld32(tB + 96, hold1);
        tc_fence_before();
        mbar_arrive(&bars[kBarBFree]);
      }
      fence_proxy_async_smem();
      named_bar(2, kDrainWarps * 32);
      if (*abort_flag) break;
      const int row = qt * kTile;
      if (issuer) {
        tma_reduce_add_4d(&P.tmap_dq, R, 0, h, row, b);
        tma_reduce_add_4d(&P.tmap_dq, R + kRBoxBytes, 32, h, row, b);
        bulk_commit_group();
        bulk_wait_read_all();
      }
      named_bar(2, kDrainWarps * 32);  // staging read: columns 64-127 next
      stage32(0, hold0);
      stage32(1, hold1);
      fence_proxy_async_smem();
      named_bar(2, kDrainWarps * 32);
      if (issuer) {
        tma_reduce_add_4d(&P.tmap_dq, R, 64, h, row, b);
        tma_reduce_add_4d(&P.tmap_dq, R + kRBoxBytes, 96, h, row, b);
        bulk_commit_group();
        bulk_wait_read_all();
      }
      named_bar(2, kDrainWarps * 32);  // staging free for the next tile
    }
    if (issuer) bulk_wait_all();
  } else if (warp < kWarpProl0 + kProlWarps) {
    // ------------------------------------------------------------ Q' / K' prologue
    const int p = tid - kWarpProl0 * 32;  // 0 .. kProlThreads - 1
    bool ok = true;
    if (phantom) {
      for (int row = p; row < kTile; row += kProlThreads) {
        zero_row(sm + kOffK, row);
        zero_row(sm + kOffV, row);
      }
    } else {
      if constexpr (QKT) ok = wait_bar(&bars[kBarKRaw], 0, abort_flag, budget);
      for (int row = p; ok && row < kTile; row += kProlThreads) {
        const int jj = kt * kTile + row;
        if constexpr (QKT) {
          if (jj < c.Skv)  // rows past S_kv stay TMA zeros
            rope_norm_inplace(sm + kOffK, row, c.wk, c.eps, c.tab16_k + b * c.tab_k_sb + (int64_t)jj * kPairs);
        } else if (jj < c.Skv) {
          rope_norm_global(c.k.p, b * c.k.sb + (int64_t)jj * c.k.ss + h * c.k.sh, c.k.is_f32, c.wk, c.eps,
                           c.tab_k + b * c.tab_k_sb + (int64_t)jj * kPairs, sm + kOffK, row);
        } else {
          zero_row(sm + kOffK, row);
        }
      }
    }
    if (ok) {
      fence_proxy_async_smem();
      mbar_arrive(&bars[kBarKFull]);
    }
    named_bar(3, kProlThreads);
    ok = !*abort_flag;  // uniform over the prologue threads
    const uint32_t peer_q = mapa_shared(smem_u32(sm + kOffQ), peer);
    const uint32_t peer_qfull = mapa_shared(smem_u32(&bars[kBarQFull]), peer);
    // Q' rows: eight lanes per row (see OctRow), four rows per warp and pass;
    // pass k of warp pw handles row 16k + 4pw + (lane & 3) of this CTA's 64.
    // The (cos, sin) rows of the next tile are loaded while this one is
    // finished, pass by pass, and pinned before the next tile starts.
    const int part = lane_id >> 2, pw = warp - kWarpProl0;
    constexpr int kPasses = kHalfRows / (kProlWarps * 4);
    auto pass_row = [&](int k) { return kHalfRows * crank + 4 * kProlWarps * k + 4 * pw + (lane_id & 3); };
    const __half2* tab16 = c.tab16_q + b * c.tab_q_sb;
    OctRow rp[kPasses];
    int m = next_pos<MK>(c, b, h, W, 0, kt0);
    if constexpr (QKT) {
      if (m < W.len) {
#pragma unroll
        for (int k = 0; k < kPasses; ++k) {
          const int i = W.qt(m) * kTile + pass_row(k);
          if (i < c.Sq) rp[k].prefetch(tab16 + (int64_t)i * kPairs, part);
        }
      }
    }
    int n = 0;
    for (; ok && m < W.len; ++n) {
      const int qt = W.qt(m);
      const int m_next = next_pos<MK>(c, b, h, W, m + 1, kt0);
      const int s = n % kQStages;
      uint8_t* tile = sm + kOffQ + s * kTileBytes;
      // LSE (base 2; +inf for rows without keys, so P = 0) and Delta of rows
      // p, p + kProlThreads, ...: every CTA keeps all 128 of the tile
      constexpr int kStatRows = kTile / kProlThreads;
      float l2[kStatRows], dl[kStatRows];
#pragma unroll
      for (int u = 0; u < kStatRows; ++u) {
        const int ii = qt * kTile + p + kProlThreads * u;
        l2[u] = INFINITY;
        dl[u] = 0.f;
        if (ii < c.Sq) {
          const int64_t ri = ((int64_t)b * c.H + h) * c.Sq + ii;
          const float l = ldg_nc_f32(P.lse + ri);
          l2[u] = (l == -INFINITY) ? INFINITY : l * kLog2e;
          dl[u] = ldg_nc_f32(P.delta + ri);
        }
      }
      // a failed wait skips the work but not the named barrier below
      if constexpr (QKT) {
        uint32_t folded = 0;
#pragma unroll
        for (int k = 0; k < kPasses; ++k) folded = rp[k].fold(folded);
        pin_loads(folded, scratch);
        if (wait_bar_warp(&bars[kBarQRaw + s], (n / kQStages) & 1, abort_flag, budget)) {
#pragma unroll
          for (int k = 0; k < kPasses; k += 2) {  // rows past S_q stay TMA zeros
            const int ra = pass_row(k), rb = pass_row(k + 1);
            OctRow::finish2(rp[k], rp[k + 1], tile, ra, rb, part, sWq, c.eps, qt * kTile + ra < c.Sq,
                            qt * kTile + rb < c.Sq);
            if (m_next < W.len) {
              const int ia = W.qt(m_next) * kTile + ra, ib = W.qt(m_next) * kTile + rb;
              if (ia < c.Sq) rp[k].prefetch(tab16 + (int64_t)ia * kPairs, part);
              if (ib < c.Sq) rp[k + 1].prefetch(tab16 + (int64_t)ib * kPairs, part);
            }
          }
        }
      } else {
        if (n < kQStages || wait_bar_cluster(&bars[kBarQFree + s], ((n / kQStages) - 1) & 1, abort_flag, budget)) {
          for (int rr = p; rr < kHalfRows; rr += kProlThreads) {  // this CTA's 64 rows
            const int row = kHalfRows * crank + rr;
            const int i = qt * kTile + row;
            if (i < c.Sq)
              rope_norm_global(c.q.p, b * c.q.sb + (int64_t)i * c.q.ss + h * c.q.sh, c.q.is_f32, c.wq, c.eps,
                               c.tab_q + b * c.tab_q_sb + (int64_t)i * kPairs, tile, row);
            else
              zero_row(tile, row);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kStatRows; ++u) {
        stat[s * 256 + p + kProlThreads * u] = l2[u];
        stat[s * 256 + 128 + p + kProlThreads * u] = dl[u];
      }
      // this CTA's 64 rows are final: one bulk copy per 64-column half to the
      // same offsets of the peer's stage, completing on its Q' barrier
      fence_proxy_async_smem();
      named_bar(3, kProlThreads);
      if (*abort_flag) break;  // uniform: set before any failed thread reached the barrier
      if (p == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t off = s * kTileBytes + hh * kHalfBytes + kHalfRowsBytes * crank;
          bulk_copy_to_peer(peer_q + off, sm + kOffQ + off, kHalfRowsBytes, peer_qfull + 8u * s);
        }
        mbar_arrive_expect_tx(&bars[kBarQFull + s], 2 * kHalfRowsBytes);  // the peer's rows
      } else {
        mbar_arrive(&bars[kBarQFull + s]);
      }
      m = m_next;
    }
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA: raw K, V, raw Q, dO
    if (lane_id == 0) {
      if (!phantom) {
        if constexpr (QKT) {
          const int y = P.k_s_first ? kt * kTile : h, z = P.k_s_first ? h : kt * kTile;
          mbar_arrive_expect_tx(&bars[kBarKRaw], kTileBytes);
          tma_load_4d(sm + kOffK, &P.tmap_k, &bars[kBarKRaw], 0, y, z, b);
          tma_load_4d(sm + kOffK + kHalfBytes, &P.tmap_k, &bars[kBarKRaw], 64, y, z, b);
        }
        const int vy = P.v_s_first ? kt * kTile : h, vz = P.v_s_first ? h : kt * kTile;
        mbar_arrive_expect_tx(&bars[kBarVFull], kTileBytes);
        tma_load_4d(sm + kOffV, &P.tmap_v, &bars[kBarVFull], 0, vy, vz, b);
        tma_load_4d(sm + kOffV + kHalfBytes, &P.tmap_v, &bars[kBarVFull], 64, vy, vz, b);
      } else {
        mbar_arrive(&bars[kBarVFull]);  // V is zeroed by the prologue, before K' is declared ready
      }
      int n = 0, q_issued = 0, lo_issued = 0, hi_issued = 0;
      for (int m = next_pos<MK>(c, b, h, W, 0, kt0); m < W.len; m = next_pos<MK>(c, b, h, W, m + 1, kt0), ++n) {
        const int qt = W.qt(m);
        const int s = n % kQStages;
        if constexpr (QKT) {  // this CTA's 64 raw rows of the tile
          if (n >= kQStages &&
              !wait_bar_cluster(&bars[kBarQFree + s], ((n / kQStages) - 1) & 1, abort_flag, budget))
            break;
          uint8_t* qrows = sm + kOffQ + s * kTileBytes + kHalfRowsBytes * crank;
          const int row = qt * kTile + kHalfRows * crank;
          const int y = P.q_s_first ? row : h, z = P.q_s_first ? h : row;
          mbar_arrive_expect_tx(&bars[kBarQRaw + s], 2 * kHalfRowsBytes);
          tma_load_4d(qrows, &P.tmap_q, &bars[kBarQRaw + s], 0, y, z, b);
          tma_load_4d(qrows + kHalfBytes, &P.tmap_q, &bars[kBarQRaw + s], 64, y, z, b);
          ++q_issued;
        }
        // dO rows [0, 64) and [64, 128) of the tile, 64-row boxes into each column half
        if (n > 0 && !wait_bar(&bars[kBarDOLoFree], (n - 1) & 1, abort_flag, budget)) break;
        {
          const int row = qt * kTile;
          const int y = P.do_s_first ? row : h, z = P.do_s_first ? h : row;
          mbar_arrive_expect_tx(&bars[kBarDOLoFull], kTileBytes / 2);
          tma_load_4d(sm + kOffDO, &P.tmap_do, &bars[kBarDOLoFull], 0, y, z, b);
          tma_load_4d(sm + kOffDO + kHalfBytes, &P.tmap_do, &bars[kBarDOLoFull], 64, y, z, b);
          ++lo_issued;
        }
        if (n > 0 && !wait_bar(&bars[kBarDOHiFree], (n - 1) & 1, abort_flag, budget)) break;
        {
          const int row = qt * kTile + 64;
          const int y = P.do_s_first ? row : h, z = P.do_s_first ? h : row;
          mbar_arrive_expect_tx(&bars[kBarDOHiFull], kTileBytes / 2);
          tma_load_4d(sm + kOffDO + kHalfBytes / 2, &P.tmap_do, &bars[kBarDOHiFull], 0, y, z, b);
          tma_load_4d(sm + kOffDO + kHalfBytes + kHalfBytes / 2, &P.tmap_do, &bars[kBarDOHiFull], 64, y, z, b);
          ++hi_issued;
        }
      }
      // drain: every issued load lands before the CTA exits (these waits do not
      // give up on abort; each is bounded)
      if (!phantom) {
        mbar_wait(&bars[kBarVFull], 0, budget);
        if constexpr (QKT) mbar_wait(&bars[kBarKRaw], 0, budget);
      }
      if (lo_issued > 0) mbar_wait(&bars[kBarDOLoFull], (lo_issued - 1) & 1, budget);
      if (hi_issued > 0) mbar_wait(&bars[kBarDOHiFull], (hi_issued - 1) & 1, budget);
      if constexpr (QKT) {
        for (int m = max(0, q_issued - kQStages); m < q_issued; ++m)
          mbar_wait(&bars[kBarQRaw + m % kQStages], (m / kQStages) & 1, budget);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue
    if (lane_id == 0) {
      constexpr uint32_t idesc_kk = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_kmn = idesc_bf16(128, 128, 0, 1);
      constexpr uint32_t idesc_mnmn = idesc_bf16(128, 128, 1, 1);
      const uint64_t dKk = sdesc_sw128(smem_u32(sm + kOffK), 16, 1024);
      const uint64_t dKm = sdesc_sw128(smem_u32(sm + kOffK), kHalfBytes, 1024);
      const uint64_t dVk = sdesc_sw128(smem_u32(sm + kOffV), 16, 1024);
      const uint64_t dOk = sdesc_sw128(smem_u32(sm + kOffDO), 16, 1024);
      const uint64_t dOm = sdesc_sw128(smem_u32(sm + kOffDO), kHalfBytes, 1024);
      const uint64_t dSk = sdesc_sw128(smem_u32(sm + kOffDS), 16, 1024);
      const uint64_t dSm = sdesc_sw128(smem_u32(sm + kOffDS), kHalfBytes, 1024);
      const uint64_t dQk0 = sdesc_sw128(smem_u32(sm + kOffQ), 16, 1024);
      const uint64_t dQm0 = sdesc_sw128(smem_u32(sm + kOffQ), kHalfBytes, 1024);
      const uint32_t tA = tmem, tB = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
      bool ok = wait_bar(&bars[kBarKFull], 0, abort_flag, budget) && wait_bar(&bars[kBarVFull], 0, abort_flag, budget);
      int m = next_pos<MK>(c, b, h, W, 0, kt0);
      int n = 0;
      bool issued = false;
      if (ok && m < W.len) {
        ok = wait_bar(&bars[kBarQFull], 0, abort_flag, budget);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tA, sdesc_add(dKk, kofs(kk)), sdesc_add(dQk0, kofs(kk)), idesc_kk, kk > 0);
          mma_commit(&bars[kBarSFull]);
          issued = true;
          ok = wait_bar(&bars[kBarDOLoFull], 0, abort_flag, budget) &&
               wait_bar(&bars[kBarDOHiFull], 0, abort_flag, budget);
        }
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tB, sdesc_add(dVk, kofs(kk)), sdesc_add(dOk, kofs(kk)), idesc_kk, kk > 0);
          mma_commit(&bars[kBarDPFull]);
        }
      }
      while (ok && m < W.len) {
        const int s = n % kQStages;
        const uint64_t dQm = sdesc_add(dQm0, s * kTileBytes);
        if (!(ok = wait_bar(&bars[kBarHalf0], n & 1, abort_flag, budget))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ts(tdV, tA + 8 * kk, sdesc_add(dOm, mofs(kk)), idesc_kmn, (n > 0 || kk > 0));
        mma_commit(&bars[kBarDOLoFree]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tdK, sdesc_add(dSk, kofs(kk)), sdesc_add(dQm, mofs(kk)), idesc_kmn, (n > 0 || kk > 0));
        if (!(ok = wait_bar(&bars[kBarHalf1], n & 1, abort_flag, budget))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 4; kk < 8; ++kk) mma_ts(tdV, tA + 64 + 8 * kk, sdesc_add(dOm, mofs(kk)), idesc_kmn, 1u);
        mma_commit(&bars[kBarDOHiFree]);
#pragma unroll
        for (int kk = 4; kk < 8; ++kk) mma_ss(tdK, sdesc_add(dSk, kofs(kk)), sdesc_add(dQm, mofs(kk)), idesc_kmn, 1u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tB, sdesc_add(dSm, mofs(kk)), sdesc_add(dKm, mofs(kk)), idesc_mnmn, kk > 0);
        mma_commit(&bars[kBarDQFull]);
        mma_commit_mc(&bars[kBarQFree + s], 0x3);  // released in both CTAs' view
        const int m_next = next_pos<MK>(c, b, h, W, m + 1, kt0);
        if (m_next < W.len) {
          const int ns = (n + 1) % kQStages;
          if (!(ok = wait_bar(&bars[kBarQFull + ns], ((n + 1) / kQStages) & 1, abort_flag, budget))) break;
          tc_fence_after();
          const uint64_t dQk = sdesc_add(dQk0, ns * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tA, sdesc_add(dKk, kofs(kk)), sdesc_add(dQk, kofs(kk)), idesc_kk, kk > 0);
          mma_commit(&bars[kBarSFull]);
          if (!(ok = wait_bar(&bars[kBarBFree], n & 1, abort_flag, budget))) break;
          if (!(ok = wait_bar(&bars[kBarDOLoFull], (n + 1) & 1, abort_flag, budget))) break;
          if (!(ok = wait_bar(&bars[kBarDOHiFull], (n + 1) & 1, abort_flag, budget))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma_ss(tB, sdesc_add(dVk, kofs(kk)), sdesc_add(dOk, kofs(kk)), idesc_kk, kk > 0);
          mma_commit(&bars[kBarDPFull]);
        }
        m = m_next;
        ++n;
      }
      if (issued && !ok) {
        // abort: let every issued MMA finish before TMEM is released
        mma_commit(&bars[kBarFinal]);
        mbar_wait(&bars[kBarFinal], 0, budget);
      }
    }
  }

  // ---- tile counters
  tc_fence_before();
  __syncthreads();
  if (!*abort_flag) {
    if (!phantom && tid == 0) {
      atomicAdd(c.counters + kCtrTilesSkipped, (unsigned long long)(c.nQt - useful));
      atomicAdd(c.counters + kCtrTilesTotal, (unsigned long long)c.nQt);
    }
  } else if (tid == 0) {
    record_timeout(c);
  }
  tc_fence_before();
  cluster_sync();  // no DSMEM store or remote arrival may target a CTA that has exited
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int MK, bool CAUSAL, bool QKT, bool ELEM>
cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  auto kern = bwd_kernel<MK, CAUSAL, QKT, ELEM>;
  static unsigned configured = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured & (1u << (dev & 31)))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
    if (e != cudaSuccess) return e;
    configured |= 1u << (dev & 31);
  }
  dim3 grid((p.c.nKt + kCluster - 1) / kCluster * kCluster, p.c.H, p.c.B);  // whole clusters
  kern<<<grid, kBwdThreads, kBwdSmem, stream>>>(p);
  return cudaGetLastError();
}

template <bool QKT>
cudaError_t launch_bwd_q(const BwdParams& p, cudaStream_t stream) {
  if (p.c.causal) return launch_bwd_t<kMaskNone, true, QKT, false>(p, stream);  // masks and causal never combine
  const bool elem = p.c.m_sq != 0;  // the mask varies along the queries
  switch (p.c.mask_kind) {
    case kMaskBool:
      return elem ? launch_bwd_t<kMaskBool, false, QKT, true>(p, stream) : launch_bwd_t<kMaskBool, false, QKT, false>(p, stream);
    case kMaskF32:
      return elem ? launch_bwd_t<kMaskF32, false, QKT, true>(p, stream) : launch_bwd_t<kMaskF32, false, QKT, false>(p, stream);
    case kMaskBF16:
      return elem ? launch_bwd_t<kMaskBF16, false, QKT, true>(p, stream) : launch_bwd_t<kMaskBF16, false, QKT, false>(p, stream);
    default: return launch_bwd_t<kMaskNone, false, QKT, false>(p, stream);
  }
}

// Kernels are specialised on the mask kind, causal masking and whether q/k
// are staged by TMA, so that each carries only its own code.
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t stream) {
  return p.qk_tma ? launch_bwd_q<true>(p, stream) : launch_bwd_q<false>(p, stream);
}

}  // namespace st
