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
//               kKStages-deep ring; bf16 rows arrive by TMA in the operand
//               layout and are normalised and rotated in place, their (cos,
//               sin) rows being fetched while the TMA is in flight (fp32 rows
//               are read from global memory, four lanes per row)
//   warp 16     TMEM allocation + tcgen05.mma issue (one thread)
//   warp 17     TMA: lane 0 raw Q and K rows, lane 1 V tiles (separate rings:
//               a K stage is released once both score MMAs of its tile are
//               done, a V stage once both PV MMAs are)
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each; P_i (bf16)
// overwrites the first 64 columns of S_i and feeds PV from TMEM.
// MMA issue order per key tile n: PV0(n-1), S0(n), PV1(n-1), S1(n), so that
// while one softmax group works on its scores the tensor core computes the
// other's. The K' ring is three tiles deep: the TMA load and the prologue of
// a key tile (several thousand cycles together) run while the MMAs of the two
// tiles before it are issued.
#include "st_common.cuh"
#include "st_kernels.h"
#include "st_prologue.cuh"

#ifndef ST_OPERAND_F16
#define ST_OPERAND_F16 false  // this unit's 16-bit operand type: bf16 (st_fwd_f16.cu: fp16)
#endif

namespace st {

namespace {

constexpr int kKStages = 3;  // K' ring: TMA load + in-place prologue run ahead of the MMAs
constexpr int kVStages = 2;
constexpr int kSoftWarps = 8;
constexpr int kWarpProl0 = 8, kProlWarps = 8;
constexpr int kWarpMma = 16, kWarpTma = 17;
constexpr int kFwdWarps = 18;
constexpr int kFwdThreads = kFwdWarps * 32;
// rescale O only when the running max grows by more than 8 (base 2); exact
// either way since O and l always share the same reference max
constexpr float kRescaleThreshold = 8.0f;
// Largest score bound (base 2) for which the fixed-reference softmax is used:
// every P = 2^(s - bound) then lies in [2^-2 bound, 1], normal in fp32 and in
// bf16 (which has fp32's exponent range; fp16 operands keep the online
// maximum, as P would fall below fp16's range).
constexpr float kFixedRefMax = 56.0f;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;                                  // 2 tiles
constexpr uint32_t kOffK = 2 * kTileBytes;                     // kKStages tiles
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;      // kVStages tiles
constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
constexpr uint32_t kOffW = kOffBar + 256;                      // q and k norm weights, fp32
constexpr uint32_t kOffFlags = kOffW + 2 * kD * 4;             // bool masks: the two query tiles' tile classes
constexpr int kMaxFlagTiles = 896;                             // key tiles whose classes fit (else read from global)
constexpr uint32_t kFwdSmem = kOffFlags + 2 * kMaxFlagTiles;   // the base must be 1024-byte aligned
static_assert(kFwdSmem <= 232448, "forward shared memory exceeds the per-block limit");

enum {
  kBarQRaw = 0,                       // raw q rows landed (TMA)
  kBarQFull,                          // + query tile (0/1): Q' ready (prologue)
  kBarQFull1,
  kBarKRaw,                           // + K stage: raw k rows landed (TMA)
  kBarKFull = kBarKRaw + kKStages,    // + K stage: K' ready (prologue)
  kBarKEmpty = kBarKFull + kKStages,  // + K stage: both score MMAs of the tile done
  kBarVFull = kBarKEmpty + kKStages,  // + V stage
  kBarVEmpty = kBarVFull + kVStages,  // + V stage: both PV MMAs of the tile done
  kBarSFull = kBarVEmpty + kVStages,  // + tile (0/1)
  kBarPFull = kBarSFull + 2,          // + tile, 128 arrivals
  kBarOFull = kBarPFull + 2,
  kNumBars = kBarOFull + 1
};
static_assert(kNumBars * 8 + 32 <= 256, "barrier area");  // + TMEM slot, abort flag, sink, K stage modes
constexpr int kBarIdProl = 1;  // named barrier of the prologue warps

// Byte offsets of K-step kk (16 elements) inside a K-major tile (two 64-column
// halves) and inside an MN-major tile (16 rows of 128 B per step); the MMA
// thread adds them to descriptors built once, so that each MMA costs it one add
// (it shares its issue slots with four busy warps).
__device__ __forceinline__ constexpr uint32_t kofs(int kk) { return (kk >> 2) * kHalfBytes + (kk & 3) * 32; }
__device__ __forceinline__ constexpr uint32_t mofs(int kk) { return kk * 2048; }

// S = Q' K'^T for one query tile: eight K-steps of 16.
template <bool F16>
__device__ __forceinline__ void issue_s(uint32_t tS, uint64_t dQ, uint64_t dK) {
  constexpr uint32_t idesc = idesc16(F16, 128, 128, 0, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) mma_ss(tS, sdesc_add(dQ, kofs(kk)), sdesc_add(dK, kofs(kk)), idesc, kk > 0);
}
// O (+)= P V with P (16-bit) in TMEM: eight K-steps of 16 keys.
template <bool F16>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint64_t dV, bool acc) {
  constexpr uint32_t idesc = idesc16(F16, 128, 128, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) mma_ts(tO, tP + kk * 8, sdesc_add(dV, mofs(kk)), idesc, acc || kk > 0);
}

// Tile classes of the CTA's two query tiles (bool masks): read from a
// shared-memory copy made at the start (when the key-tile count fits), since
// the MMA thread consults them on its critical path, else from global memory.
struct PairFlags {
  const uint8_t* sm;  // [2][kMaxFlagTiles] or nullptr
  const uint8_t* g0;  // global rows of the two query tiles
  const uint8_t* g1;
  bool has1;          // the second query tile exists (the last pair may have one tile)
};

template <int MK>
__device__ __forceinline__ uint8_t tile_flag(const PairFlags& f, int ti, int kt) {
  if (ti && !f.has1) return kTileAllFalse;
  if constexpr (MK == kMaskBool) {
    if (f.sm) return f.sm[ti * kMaxFlagTiles + kt];
    return (ti ? f.g1 : f.g0)[kt];
  }
  if constexpr (MK == kMaskNone) return kTileAllTrue;
  return kTileMixed;  // additive masks are always applied
}

__device__ __forceinline__ float c_wq(const Common& c, int d) { return __ldg(c.wq + d); }
__device__ __forceinline__ float c_wk(const Common& c, int d) { return __ldg(c.wk + d); }

// The CTA's walk over its key tiles [0, L): position u visits tile
// (u + rot) mod L. The CTAs of a head start at evenly spread tiles, so that a
// K' tile one of them publishes is usually in place before the others reach
// it (the online softmax does not depend on the order).
struct KWalk {
  int L, rot;
  __device__ __forceinline__ int tile(int u) const { return u + rot >= L ? u + rot - L : u + rot; }
};

// Next walk position at or after u whose tile at least one of the two query
// tiles needs.
template <int MK>
__device__ __forceinline__ int next_tile(const PairFlags& f, const KWalk& w, int u) {
  if constexpr (MK == kMaskBool) {
    for (; u < w.L; ++u) {
      const int kt = w.tile(u);
      if (tile_flag<MK>(f, 0, kt) != kTileAllFalse || tile_flag<MK>(f, 1, kt) != kTileAllFalse) break;
    }
  }
  return u;
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

template <int MK, bool CAUSAL, bool QKT, bool F16>
__device__ __forceinline__ void fwd_body(const FwdParams& P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_u32(sm) & 1023u) {  // the layout has no slack: refuse an unaligned base (uniform over the grid)
    if (threadIdx.x == 0) atomicOr(P.c.status, kStatusLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  // per K stage: 1 when the stage received a finished K' tile from the
  // workspace (another CTA published it), 0 when the prologue builds it
  volatile uint32_t* kmode = tslot + 4;

  const Common& c = P.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
  const int pair = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / P.c.group;  // the K/V head of query head h (grouped K/V heads)
  const int qt0 = 2 * pair;

  if (warp == kWarpMma) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars[kBarQRaw], 1);
    mbar_init(&bars[kBarQFull + 0], kProlWarps * 32);
    mbar_init(&bars[kBarQFull + 1], kProlWarps * 32);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars[kBarKRaw + s], 1);
      mbar_init(&bars[kBarKFull + s], kProlWarps * 32);
      mbar_init(&bars[kBarKEmpty + s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars[kBarVFull + s], 1);
      mbar_init(&bars[kBarVEmpty + s], 1);
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
  PairFlags fl{nullptr, nullptr, nullptr, qt0 + 1 < c.nQt};
  if constexpr (MK == kMaskBool) {
    const uint8_t* row = c.flags + b * c.f_sb + h * c.f_sh;
    fl.g0 = row + qt0 * c.f_sq;
    fl.g1 = fl.has1 ? row + (qt0 + 1) * c.f_sq : fl.g0;
    if (c.nKt <= kMaxFlagTiles) {
      uint8_t* sf = sm + kOffFlags;
      for (int e = tid; e < 2 * c.nKt; e += kFwdThreads) {
        const int ti = e >= c.nKt, kt = e - ti * c.nKt;
        sf[ti * kMaxFlagTiles + kt] = (ti ? fl.g1 : fl.g0)[kt];
      }
      fl.sm = sf;
    }
  }
  if (warp == kWarpTma && lane_id == 0) {
    tma_prefetch_desc(&P.tmap_v);
    if (P.save_qp) tma_prefetch_desc(&P.tmap_qp);
    if (P.kcache) tma_prefetch_desc(&P.tmap_kc);
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
  KWalk kw;
  kw.L = kt_end;
  kw.rot = kt_end > 0 ? static_cast<int>((static_cast<int64_t>(pair) * kt_end) / gridDim.x) : 0;
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
    // Fixed-reference softmax. The operands are RMS-normalised rows scaled by
    // the norm weights and rotated, so |q'| <= sqrt(D) max|w_q| and
    // |k'| <= sqrt(D) max|w_k|, and every score obeys
    //   |s * scale * log2(e)| <= bound = scale * log2(e) * D * max|w_q| * max|w_k|
    // (times 1.02 for the rounding of q', k' to the 16-bit operand type). When
    // the mask adds no values (none, bool, causal) and the bound is small
    // enough, P = 2^(s * scale * log2(e) - bound) needs no row maximum: one
    // pass over the scores, no rescaling of O; LSE = bound + log2(l). (Softmax
    // is invariant to the reference; only its range matters.)
    float fixed_ref = INFINITY;
    if constexpr ((MK == kMaskNone || MK == kMaskBool) && !F16) {
      float wq_m = 0.f, wk_m = 0.f;
#pragma unroll
      for (int d = lane_id; d < kD; d += 32) {
        wq_m = fmaxf(wq_m, fabsf(sW[d]));
        wk_m = fmaxf(wk_m, fabsf(sW[kD + d]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        wq_m = fmaxf(wq_m, __shfl_xor_sync(0xffffffffu, wq_m, o));
        wk_m = fmaxf(wk_m, __shfl_xor_sync(0xffffffffu, wk_m, o));
      }
      const float bound = sc * static_cast<float>(kD) * wq_m * wk_m * 1.02f;
      if (bound <= kFixedRefMax) fixed_ref = bound;  // the same decision in every thread (same weights)
    }
    const bool fixed = fixed_ref != INFINITY;
    float m_run = fixed ? fixed_ref : -INFINITY, l_run = 0.f;
    int n = 0, useful = 0;
    bool ok = true;
    for (int u = next_tile<MK>(fl, kw, 0); u < kw.L; u = next_tile<MK>(fl, kw, u + 1), ++n) {
      const int kt = kw.tile(u);
      const uint8_t flag = tile_flag<MK>(fl, ti, kt);
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
      if (fixed) {
        // one pass: P = exp2(s - bound) (16-bit, into the first 64 S columns), row sum
        float ls0 = 0.f, ls1 = 0.f;
        if (plain) {
          uint32_t ra[16], rb[16];
          const float2 sc2 = make_float2(sc, sc), nb2 = make_float2(-fixed_ref, -fixed_ref);
          float2 ls = make_float2(0.f, 0.f);
          tmem_ld16_issue(tS, ra);
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {
            uint32_t(&cur)[16] = (q8 & 1) ? rb : ra;
            uint32_t(&nxt)[16] = (q8 & 1) ? ra : rb;
            tmem_ld_wait16(cur);
            if (q8 < 7) tmem_ld16_issue(tS + 16 * (q8 + 1), nxt);
            uint32_t pw[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(cur[2 * t]), __uint_as_float(cur[2 * t + 1])), sc2, nb2);
              const float p0 = ex2(x.x), p1 = ex2(x.y);
              ls = __fadd2_rn(ls, make_float2(p0, p1));
              pw[t] = pack16<F16>(p0, p1);
            }
            tmem_st8(tS + 8 * q8, pw);
          }
          ls0 = ls.x;
          ls1 = ls.y;
        } else {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t raw[32], pw[16];
            tmem_ld32(tS + 32 * q4, raw);
            float sv[32];
            masked_scores32<MK, CAUSAL>(c, raw, b, h, i, j0 + 32 * q4, flag, mbits[q4], sv, mask_vec, scratch);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const float p0 = ex2(sv[2 * t] - fixed_ref), p1 = ex2(sv[2 * t + 1] - fixed_ref);
              ls0 += p0;
              ls1 += p1;
              pw[t] = pack16<F16>(p0, p1);
            }
            tmem_st16(tS + 16 * q4, pw);  // over columns this step or an earlier one has read
          }
        }
        l_run += ls0 + ls1;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[kBarPFull + ti]);
        continue;
      }
      // pass 1: row max (raw scores on plain tiles; the scale is positive)
      float mt = -INFINITY;
      if (plain) {
        // each 16-column load is issued before the previous one is reduced
        uint32_t ra[16], rb[16];
        float m0 = -INFINITY, m1 = -INFINITY;
        tmem_ld16_issue(tS, ra);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          uint32_t(&cur)[16] = (q8 & 1) ? rb : ra;
          uint32_t(&nxt)[16] = (q8 & 1) ? ra : rb;
          tmem_ld_wait16(cur);
          if (q8 < 7) tmem_ld16_issue(tS + 16 * (q8 + 1), nxt);
#pragma unroll
          for (int t = 0; t < 16; t += 4) {
            m0 = fmax3(m0, __uint_as_float(cur[t]), __uint_as_float(cur[t + 1]));
            m1 = fmax3(m1, __uint_as_float(cur[t + 2]), __uint_as_float(cur[t + 3]));
          }
        }
        mt = fmaxf(m0, m1) * sc;
      }
      if (!plain) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t raw[32];
          tmem_ld32(tS + 32 * q4, raw);
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
        tmem_st_wait();
      }
      float corr = 1.f;
      if (mt > m_run + kRescaleThreshold || (m_run == -INFINITY && mt > -INFINITY)) {
        corr = ex2(m_run - mt);  // 0 when m_run is -inf
        m_run = mt;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // pass 2: P = exp2(s - m) (bf16 into the first 64 S columns), row sum.
      // Step q8 of P lands in columns [8 q8, 8 q8 + 8), which the loads of
      // steps <= q8 have already read.
      float ls0 = 0.f, ls1 = 0.f;
      if (plain) {
        uint32_t ra[16], rb[16];
        const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_use, -m_use);
        float2 ls = make_float2(0.f, 0.f);
        tmem_ld16_issue(tS, ra);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          uint32_t(&cur)[16] = (q8 & 1) ? rb : ra;
          uint32_t(&nxt)[16] = (q8 & 1) ? ra : rb;
          tmem_ld_wait16(cur);
          if (q8 < 7) tmem_ld16_issue(tS + 16 * (q8 + 1), nxt);
          uint32_t pw[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(cur[2 * t]), __uint_as_float(cur[2 * t + 1])), sc2, nm2);
            const float p0 = ex2(x.x), p1 = ex2(x.y);
            ls = __fadd2_rn(ls, make_float2(p0, p1));
            pw[t] = pack16<F16>(p0, p1);
          }
          tmem_st8(tS + 8 * q8, pw);
        }
        ls0 = ls.x;
        ls1 = ls.y;
      }
      if (!plain) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t raw[32], pw[16];
          tmem_ld32(tS + 32 * q4, raw);
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float p0 = ex2(__uint_as_float(raw[2 * t]) - m_use), p1 = ex2(__uint_as_float(raw[2 * t + 1]) - m_use);
            ls0 += p0;
            ls1 += p1;
            pw[t] = pack16<F16>(p0, p1);
          }
          tmem_st16(tS + 16 * q4, pw);
        }
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
        if (i < c.Sq) store_chunk32(P.o, ooff, P.o_dt, q4, y);
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
          HalfRowPrologue<F16> hp;
          if (i < c.Sq) {
            const __half2* t16 = c.tab16_q + b * c.tab_q_sb + (int64_t)i * kPairs;
            hp.prefetch(t16, hh);
            hp.prefetch2(t16, hh);
          }
          hp.finish(tile, prow, hh, sW, c.eps, i < c.Sq);
        } else {
          // fp32 rows from global memory, four lanes per row (every prologue
          // thread in every pass: the row's sum of squares is a shuffle)
#pragma unroll 1
          for (int pass = 0; pass < kTile * 4 / (kProlWarps * 32); ++pass) {
            const int row = pass * (kProlWarps * 8) + (p >> 2), i = (qt0 + ti) * kTile + row;
            const bool valid = i < c.Sq;
            const int iv = valid ? i : 0;
            rope_norm_global_quad<F16>(c.q.p, b * c.q.sb + (int64_t)iv * c.q.ss + h * c.q.sh, c.q.dt, c.wq, c.eps,
                                       c.tab_q + b * c.tab_q_sb + (int64_t)iv * kPairs, tile, row, p & 3, valid,
                                       kHalfBytes);
          }
        }
        // each tile is released as soon as it is final: S0 of the first key
        // tile does not wait for the second query tile
        fence_proxy_async_smem();
        mbar_arrive(&bars[kBarQFull + ti]);
      }
    }
    // one decision for the prologue warps, which share a named barrier below
    ok = !named_bar_any(kBarIdProl, kProlWarps * 32, !ok);
    // K' tiles: built here unless another CTA of the same head already
    // published the tile in the workspace (the TMA warp then loaded it
    // finished). A tile built here is published in turn: thread 0 stores it by
    // TMA and, once the store has completed, raises the tile's flag (release);
    // the flag of one tile is raised when the next one is published or at the
    // end, so the wait for completion never stalls a tile.
    const uint32_t* flag_row = P.kflags + ((int64_t)b * c.Hkv + hk) * c.nKt;
    int pend_kt = -1;  // thread 0: the tile whose store is in flight
    auto raise_pending = [&]() {
      if (pend_kt < 0) return;
      bulk_wait_all();
      fence_proxy_async_global();
      st_release_gpu(const_cast<uint32_t*>(flag_row) + pend_kt, 1u);
      pend_kt = -1;
    };
    int n = 0;
    for (int u = next_tile<MK>(fl, kw, 0); ok && u < kw.L; u = next_tile<MK>(fl, kw, u + 1), ++n) {
      const int kt = kw.tile(u);
      const int slot = n % kKStages;
      uint8_t* tile = sm + kOffK + slot * kTileBytes;
      // the stage is free and its rows (raw, or a published K' tile) have
      // landed; fp32 rows are read from global memory below
      const bool got = wait_bar_warp(&bars[kBarKRaw + slot], (n / kKStages) & 1, abort_flag, budget);
      const bool cached = got && kmode[slot] != 0u;
      if (got && !cached) {
        if constexpr (QKT) {
          const int j = kt * kTile + prow;
          HalfRowPrologue<F16> hp;
          if (j < c.Skv) {
            const __half2* t16 = c.tab16_k + b * c.tab_k_sb + (int64_t)j * kPairs;
            hp.prefetch(t16, hh);
            hp.prefetch2(t16, hh);
          }
          hp.finish(tile, prow, hh, sW + kD, c.eps, j < c.Skv);
        } else {
#pragma unroll 1
          for (int pass = 0; pass < kTile * 4 / (kProlWarps * 32); ++pass) {
            const int row = pass * (kProlWarps * 8) + (p >> 2), j = kt * kTile + row;
            const bool valid = j < c.Skv;
            const int jv = valid ? j : 0;
            rope_norm_global_quad<F16>(c.k.p, b * c.k.sb + (int64_t)jv * c.k.ss + hk * c.k.sh, c.k.dt, c.wk, c.eps,
                                       c.tab_k + b * c.tab_k_sb + (int64_t)jv * kPairs, tile, row, p & 3, valid,
                                       kHalfBytes);
          }
        }
        fence_proxy_async_smem();
      }
      if (P.kcache) {
        if (named_bar_any(kBarIdProl, kProlWarps * 32, !got)) break;  // the tile's rows are final
        if (!cached && p == 0) {
          raise_pending();
          tma_store_4d(&P.tmap_kc, tile, 0, hk, kt * kTile, b);  // rows past S_kv are clipped
          tma_store_4d(&P.tmap_kc, tile + kHalfBytes, 64, hk, kt * kTile, b);
          bulk_commit_group();
          bulk_wait_read_all();  // read before the stage can be released and refilled
          pend_kt = kt;
        }
      } else if (!got) {
        break;
      }
      mbar_arrive(&bars[kBarKFull + slot]);
    }
    if (p == 0) raise_pending();
    // the backward's dQ' accumulator rows of this CTA's queries start at zero
    // (a backward that reuses this workspace skips its own zeroing pass): one
    // 512-byte row per warp instruction
    if (ok && P.dq_zero) {
      const int pw = p >> 5;
#pragma unroll 1
      for (int rr = pw; rr < 2 * kTile; rr += kProlWarps) {
        const int i = qt0 * kTile + rr;
        if (i >= c.Sq) break;
        reinterpret_cast<float4*>(P.dq_zero + (((int64_t)b * c.Sq + i) * c.H + h) * kD)[lane_id] =
            make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA: raw Q, raw K (lane 0), V (lane 1)
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
      // the K ring: a published K' tile (finished, from the workspace), else
      // the raw 16-bit rows (normalised in place by the prologue), else (fp32
      // rows, which the prologue reads itself) a plain arrival
      const uint32_t* flag_row = P.kflags + ((int64_t)b * c.Hkv + hk) * c.nKt;
      int n = 0;
      for (int u = next_tile<MK>(fl, kw, 0); u < kw.L; u = next_tile<MK>(fl, kw, u + 1), ++n) {
        const int kt = kw.tile(u);
        const int slot = n % kKStages;
        if (n >= kKStages && !wait_bar(&bars[kBarKEmpty + slot], ((n / kKStages) - 1) & 1, abort_flag, budget))
          break;
        uint8_t* ktile = sm + kOffK + slot * kTileBytes;
        const bool cached = P.kcache && ld_acquire_gpu(flag_row + kt) != 0u;
        kmode[slot] = cached ? 1u : 0u;
        if (cached) {
          fence_proxy_async_global();  // the TMA read is ordered after the flag
          mbar_arrive_expect_tx(&bars[kBarKRaw + slot], kTileBytes);
          tma_load_4d(ktile, &P.tmap_kc, &bars[kBarKRaw + slot], 0, hk, kt * kTile, b);
          tma_load_4d(ktile + kHalfBytes, &P.tmap_kc, &bars[kBarKRaw + slot], 64, hk, kt * kTile, b);
        } else if constexpr (QKT) {
          const int y = P.k_s_first ? kt * kTile : hk, z = P.k_s_first ? hk : kt * kTile;
          mbar_arrive_expect_tx(&bars[kBarKRaw + slot], kTileBytes);
          tma_load_4d(ktile, &P.tmap_k, &bars[kBarKRaw + slot], 0, y, z, b);
          tma_load_4d(ktile + kHalfBytes, &P.tmap_k, &bars[kBarKRaw + slot], 64, y, z, b);
        } else {
          mbar_arrive(&bars[kBarKRaw + slot]);
        }
      }
      // every issued load lands before the CTA exits (these waits do not
      // give up on abort; each is bounded)
      if constexpr (QKT) mbar_wait(&bars[kBarQRaw], 0, budget);
      for (int m = max(0, n - kKStages); m < n; ++m)
        mbar_wait(&bars[kBarKRaw + m % kKStages], (m / kKStages) & 1, budget);
    } else if (lane_id == 1) {
      int n = 0;
      for (int u = next_tile<MK>(fl, kw, 0); u < kw.L; u = next_tile<MK>(fl, kw, u + 1), ++n) {
        const int kt = kw.tile(u);
        const int slot = n % kVStages;
        if (n >= kVStages && !wait_bar(&bars[kBarVEmpty + slot], ((n / kVStages) - 1) & 1, abort_flag, budget)) break;
        uint8_t* tile = sm + kOffV + slot * kTileBytes;
        const int y = P.v_s_first ? kt * kTile : hk, z = P.v_s_first ? hk : kt * kTile;
        mbar_arrive_expect_tx(&bars[kBarVFull + slot], kTileBytes);
        tma_load_4d(tile, &P.tmap_v, &bars[kBarVFull + slot], 0, y, z, b);
        tma_load_4d(tile + kHalfBytes, &P.tmap_v, &bars[kBarVFull + slot], 64, y, z, b);
      }
      for (int m = max(0, n - kVStages); m < n; ++m)
        mbar_wait(&bars[kBarVFull + m % kVStages], (m / kVStages) & 1, budget);
    } else if (lane_id == 2 && P.save_qp) {
      // the finished Q' tiles go to the workspace for the backward (rows past
      // S_q are clipped by the map); the tiles stay in place for the whole CTA
      if (wait_bar(&bars[kBarQFull + 0], 0, abort_flag, budget) && wait_bar(&bars[kBarQFull + 1], 0, abort_flag, budget)) {
#pragma unroll 1
        for (int ti = 0; ti < 2; ++ti) {
          const int row = (qt0 + ti) * kTile;
          if (row >= c.Sq) break;
          const uint8_t* tile = sm + kOffQ + ti * kTileBytes;
          tma_store_4d(&P.tmap_qp, tile, 0, h, row, b);
          tma_store_4d(&P.tmap_qp, tile + kHalfBytes, 64, h, row, b);
        }
        bulk_commit_group();
        bulk_wait_read_all();  // the source tiles are read before the CTA may exit
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue
    if (lane_id == 0) {
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + kOffQ), 16, 1024), dQ1 = sdesc_add(dQ0, kTileBytes);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sm + kOffK), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sm + kOffV), kHalfBytes, 1024);
      const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
      int u = next_tile<MK>(fl, kw, 0);  // walk position (the MMAs need no tile index)
      int n = 0;
      bool issued = false;
      bool ok = true;
      if (u < kw.L) {
        ok = wait_bar(&bars[kBarQFull + 0], 0, abort_flag, budget) &&
             wait_bar(&bars[kBarKFull + 0], 0, abort_flag, budget);
        if (ok) {
          tc_fence_after();
          issue_s<F16>(tS0, dQ0, dK0);
          mma_commit(&bars[kBarSFull + 0]);
          issued = true;
          if ((ok = wait_bar(&bars[kBarQFull + 1], 0, abort_flag, budget))) {
            tc_fence_after();
            issue_s<F16>(tS1, dQ1, dK0);
            mma_commit(&bars[kBarSFull + 1]);
            mma_commit(&bars[kBarKEmpty + 0]);
          }
        }
      }
      while (ok && u < kw.L) {
        const int vslot = n % kVStages;
        const int u_next = next_tile<MK>(fl, kw, u + 1);
        const bool has_next = u_next < kw.L;
        const int nslot = (n + 1) % kKStages;
        const uint64_t dV = sdesc_add(dV0, vslot * kTileBytes), dK = sdesc_add(dK0, nslot * kTileBytes);
        if (!(ok = wait_bar(&bars[kBarVFull + vslot], (n / kVStages) & 1, abort_flag, budget))) break;
        if (!(ok = wait_bar(&bars[kBarPFull + 0], n & 1, abort_flag, budget))) break;
        tc_fence_after();
        issue_pv<F16>(tO0, tS0, dV, n > 0);
        if (has_next) {
          if (!(ok = wait_bar(&bars[kBarKFull + nslot], ((n + 1) / kKStages) & 1, abort_flag, budget))) break;
          tc_fence_after();
          issue_s<F16>(tS0, dQ0, dK);
          mma_commit(&bars[kBarSFull + 0]);
        }
        if (!(ok = wait_bar(&bars[kBarPFull + 1], n & 1, abort_flag, budget))) break;
        tc_fence_after();
        issue_pv<F16>(tO1, tS1, dV, n > 0);
        mma_commit(&bars[kBarVEmpty + vslot]);
        if (has_next) {
          issue_s<F16>(tS1, dQ1, dK);
          mma_commit(&bars[kBarSFull + 1]);
          mma_commit(&bars[kBarKEmpty + nslot]);
        }
        u = u_next;
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

  // the lanes of the single-thread roles wait for their lane 0 here, at a warp
  // barrier, rather than at the block barrier below
  __syncwarp();
  if (*abort_flag && tid == 0) record_timeout(c);
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

template <int MK, bool CAUSAL, bool QKT, bool F16>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams P) {
  grid_dependency_wait();
  if constexpr (MK == kMaskBool) {
    // A bool mask whose every element is True (found by the classify kernel,
    // which completed before the wait above) masks nothing: the unmasked
    // kernel body computes the same results without the per-tile class
    // lookups.
    if (*P.c.mask_any_false == 0u) {
      fwd_body<kMaskNone, CAUSAL, QKT, F16>(P);
      return;
    }
  }
  fwd_body<MK, CAUSAL, QKT, F16>(P);
}

}  // namespace

template <int MK, bool CAUSAL, bool QKT, bool F16>
cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_kernel<MK, CAUSAL, QKT, F16>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = opt_in_smem(kern, kFwdSmem, configured);
  if (e != cudaSuccess) return e;
  dim3 grid((p.c.nQt + 1) / 2, p.c.H, p.c.B);
  return launch_chained(kern, grid, dim3(kFwdThreads), kFwdSmem, stream, p);
}

template <bool QKT, bool F16>
cudaError_t launch_fwd_q(const FwdParams& p, cudaStream_t stream) {
  if (p.c.causal) return launch_fwd_t<kMaskNone, true, QKT, F16>(p, stream);  // masks and causal never combine
  switch (p.c.mask_kind) {
    case kMaskBool: return launch_fwd_t<kMaskBool, false, QKT, F16>(p, stream);
    case kMaskF32: return launch_fwd_t<kMaskF32, false, QKT, F16>(p, stream);
    case kMaskBF16: return launch_fwd_t<kMaskBF16, false, QKT, F16>(p, stream);
    default: return launch_fwd_t<kMaskNone, false, QKT, F16>(p, stream);
  }
}

// Kernels are specialised on the mask kind, causal masking, whether q/k are
// staged by TMA and the 16-bit operand type, so that each carries only its
// own code. This translation unit holds one operand type (ST_OPERAND_F16).
#if ST_OPERAND_F16
cudaError_t launch_fwd_f16(const FwdParams& p, cudaStream_t stream) {
#else
cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream) {
#endif
  return p.qk_tma ? launch_fwd_q<true, ST_OPERAND_F16>(p, stream) : launch_fwd_q<false, ST_OPERAND_F16>(p, stream);
}

}  // namespace st
