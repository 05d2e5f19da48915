// Backward main kernel: one CTA per (key tile of 128 rows, K/V head, batch),
// in clusters of two CTAs over adjacent key tiles (kt0 = 2p, kt0 + 1) that
// walk the same query tiles in lockstep, for every query head that shares the
// K/V head (grouped K/V heads: dK' and dV accumulate over the whole group in
// TMEM, so dk and dv leave the epilogue final). Per query tile of 128 rows,
// with Q' = RoPE(RMSNorm(q)) and K' the same for k (16-bit, 128B-swizzled
// operand tiles):
//   S^T = K' Q'^T, dP^T = V dO^T                      (tensor core, TMEM)
//   P^T = exp2(S^T scale log2e - LSE log2e)            (compute warps)
//   dS^T = P^T (dP^T - Delta)
//   dV += P^T dO, dK' += dS^T Q', dQ'^T = K'^T dS^T    (tensor core, TMEM)
// Every MMA is M = 128, N = 128: a tcgen05 MMA with N = 64 takes as long as
// one with N = 128 (measured on GB300: 64 cycles per K-step either way), so
// whole 128-query tiles keep the tensor core at its full rate. dQ'^T (this
// CTA's 128 keys) is added into a global fp32 accumulator by TMA bulk
// reduces. Q' comes from the workspace, where the forward kernel left the
// tiles it normalised and rotated (a standalone row kernel fills it when the
// forward did not run on this workspace); each CTA of a cluster loads half of
// a tile's rows by TMA multicast into both CTAs' stage.
//
// Warp roles (608 threads; 96 registers per thread):
//   warps 0-7    compute: warp w owns TMEM lanes 32*(w%4).. (key rows) and
//                queries [64*(w/4), +64) of each tile, in two 32-query chunks;
//                P^T goes to TMEM (16-bit, inside the chunk's own S^T
//                columns), dS^T to shared memory
//   warps 8-11   dQ drain: TMEM lanes = head dims; a tile's dQ'^T is read out
//                in two 64-query halves and its columns released; each warp
//                stages its 32 head dims as a [64 query][32] box in the tile's
//                (then idle) dO stage and adds it into global memory with a TMA
//                bulk reduce of its own
//   warps 12-15  prologue: K' once (normalised and rotated in place); then
//                each tile's LSE and Delta
//   warp 16      TMEM allocation + tcgen05.mma issue (one thread)
//   warp 17      TMA: raw K, V once; this CTA's 64 Q' rows per tile,
//                multicast to both CTAs (2-stage ring, a stage reused once both
//                CTAs' MMAs released it)
//   warp 18      TMA: dO tiles (2-stage ring)
// TMEM (512 columns): X = S^T (later P^T), Y = dP^T (later dQ'^T), dV, dK',
// 128 columns each.
// MMA order for tile n: [P^T(n) in TMEM] dV, S^T(n+1) over P^T(n) (the dV
// MMAs read it first: same issuing thread, in order) | [dS^T(n) in shared
// memory] dQ'^T(n) over dP^T(n), dK' | [dQ'^T(n) drained] dP^T(n+1). The
// compute warps build P^T(n+1) while the tensor core finishes tile n, and keep
// it in registers for dS^T(n+1), since S^T(n+2) overwrites it in TMEM.
#include "st_common.cuh"
#include "st_kernels.h"
#include "st_prologue.cuh"

#ifndef ST_OPERAND_F16
#define ST_OPERAND_F16 false  // this unit's 16-bit operand type: bf16 (st_bwd_f16.cu: fp16)
#endif

namespace st {

namespace {

constexpr int kCluster = 2;
constexpr int kComputeWarps = 8;
constexpr int kWarpDrain0 = 8, kDrainWarps = 4;
constexpr int kWarpProl0 = 12, kProlWarps = 4;
constexpr int kWarpMma = 16, kWarpTma = 17, kWarpTmaDO = 18;
constexpr int kBwdWarps = 19;
constexpr int kBwdThreads = kBwdWarps * 32;
constexpr int kProlThreads = kProlWarps * 32;
constexpr int kQStages = 2;                                // Q' ring, in tiles
constexpr int kDOStages = 2;                               // dO ring, in tiles
constexpr uint32_t kQTileBytes = kTile * kD * 2;           // 32 KB 16-bit tile (two 16 KB column halves)
constexpr int kPeerRows = kTile / kCluster;                // Q' rows produced per CTA per tile
constexpr uint32_t kPeerRowsBytes = kPeerRows * 128;       // those rows in one column half
constexpr int kDrainRows = 64;                             // queries per drain box (the dQ map's box)
constexpr uint32_t kRBoxBytes = kDrainRows * 32 * 4;       // one [64 queries][32 head dims] fp32 box
// named barrier of the epilogue: the compute, drain and prologue warps (16)
constexpr int kBarIdEpi = 4, kEpiThreads = (kComputeWarps + kDrainWarps + kProlWarps) * 32;
static_assert(kComputeWarps + kDrainWarps + kProlWarps == 16 && kWarpProl0 + kProlWarps == kWarpMma,
              "the epilogue warps are warps 0-15: four per TMEM lane quarter");
constexpr uint32_t kBoxBytes = 128 * 128;                  // a [128 rows][128 bytes] TMA box

// shared memory layout (offsets from the 1024-byte aligned dynamic base)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kTileBytes;
constexpr uint32_t kOffQ = 2 * kTileBytes;                      // kQStages tiles
constexpr uint32_t kOffDO = kOffQ + kQStages * kQTileBytes;     // kDOStages tiles
constexpr uint32_t kOffDS = kOffDO + kDOStages * kQTileBytes;   // [128 keys][128 queries] 16-bit
constexpr uint32_t kOffStat = kOffDS + kQTileBytes;             // [stage][LSE*log2e | Delta][128] fp32
constexpr uint32_t kOffBar = kOffStat + kQStages * 2 * kTile * 4;
constexpr uint32_t kBarBytes = 512;
constexpr uint32_t kOffW = kOffBar + kBarBytes;                 // k norm weights for the epilogue, fp32
constexpr uint32_t kBwdSmem = kOffW + kD * 4;                   // the base must be 1024-byte aligned
static_assert(kBwdSmem <= 232448, "backward shared memory exceeds the per-block limit");
static_assert(kProlThreads >= kTile, "one prologue thread per stat row");
static_assert(kDrainWarps * kRBoxBytes <= kQTileBytes, "the drain boxes fit in a dO stage");
static_assert(kQStages * 2 * kTile >= 4 * kTile, "the epilogue's row-sum exchange fits in the stat area");
static_assert(kDOStages >= 2, "the epilogue stages dV in the first dO stage and a row-sum exchange in the second");

enum {
  kBarKRaw = 0,                          // raw k rows landed (TMA)
  kBarKFull,                             // K' ready (and V, for a CTA past the last key tile)
  kBarVFull,
  kBarQRaw,                              // + stage: Q' rows landed (both CTAs' multicast loads)
  kBarQFull = kBarQRaw + kQStages,       // + stage: the stage's LSE/Delta written (prologue threads)
  kBarQFree = kBarQFull + kQStages,      // + stage: both CTAs' MMAs done with the stage
  kBarDOFull = kBarQFree + kQStages,     // + stage: dO rows landed
  kBarDOFree = kBarDOFull + kDOStages,   // + stage: MMAs done with the dO rows, drain boxes read
  kBarSFull = kBarDOFree + kDOStages,    // S^T in TMEM
  kBarDPFull,                            // dP^T in TMEM
  kBarPDone,                             // P^T in TMEM (256 arrivals)
  kBarCDone,                             // dS^T in shared memory, dP^T read (256 arrivals)
  kBarDQ,                                // dQ'^T in TMEM (and every earlier MMA done)
  kBarBFree,                             // dQ'^T read out (128 arrivals)
  kBarFinal,                             // every issued MMA done (end of the walk, or abort)
  kBarEpi,                               // epilogue: raw k rows and (cos, sin) rows staged
  kNumBars
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");  // + TMEM slot, abort flag, sink, K tile mode

__device__ __forceinline__ uint32_t kofs128(int kk) { return (kk >> 2) * kHalfBytes + (kk & 3) * 32; }  // K-major, 128 rows
__device__ __forceinline__ uint32_t mofs(int kk) { return kk * 2048; }                                   // MN-major, 16 rows
// TMEM columns: X holds S^T and then P^T, Y dP^T and then dQ'^T
constexpr uint32_t kColX = 0, kColY = 128, kColDV = 256, kColDK = 384;
// P^T of queries 32 c .. 32 c + 31 (chunk c of the tile) is packed, two
// 16-bit values per column, into the first 16 of the chunk's 32 S^T columns:
// the A operand of K-step kk (queries 16 kk ..) starts at this column of X.
__device__ __forceinline__ uint32_t p_col(int kk) { return 32 * (kk >> 1) + 8 * (kk & 1); }

// Tile class of (query tile qt, key tile kt) for this CTA's own key tile; a
// CTA past the last key tile sees nothing.
template <int MK>
__device__ __forceinline__ uint8_t own_flag(const Common& c, int b, int h, int qt, int kt) {
  if (kt >= c.nKt) return kTileAllFalse;
  if constexpr (MK == kMaskBool) return c.flags[b * c.f_sb + h * c.f_sh + qt * c.f_sq + kt];
  if constexpr (MK == kMaskNone) return kTileAllTrue;
  return kTileMixed;
}

// What a cluster visits: for each query head h0 .. h0 + group - 1 that shares
// its K/V head (grouped K/V heads; group = 1 otherwise), the query tiles
// [begin, begin + len), walked from a rotated start so that the clusters of
// one head (which all add into the same dQ rows) do not work on the same query
// tile at the same time. A position is (g, mm): step mm of the walk of head
// h0 + g; every role steps through it without divisions.
struct WPos {
  int g, mm;
};
struct QWalk {
  int begin, len, rot, h0, group;
  __device__ __forceinline__ WPos start() const { return WPos{len > 0 ? 0 : group, 0}; }
  __device__ __forceinline__ bool more(const WPos& p) const { return p.g < group; }
  __device__ __forceinline__ WPos step(WPos p) const {
    if (++p.mm == len) {
      p.mm = 0;
      ++p.g;
    }
    return p;
  }
  __device__ __forceinline__ int qt(const WPos& p) const {
    const int x = rot + p.mm;
    return begin + (x >= len ? x - len : x);
  }
  __device__ __forceinline__ int head(const WPos& p) const { return h0 + p.g; }
};

// Next walk position at or after p whose query tile either key tile of the
// cluster needs.
template <int MK>
__device__ __forceinline__ WPos next_pos(const Common& c, int b, const QWalk& w, WPos p, int kt0) {
  if constexpr (MK == kMaskBool) {
    while (w.more(p) && own_flag<MK>(c, b, w.head(p), w.qt(p), kt0) == kTileAllFalse &&
           own_flag<MK>(c, b, w.head(p), w.qt(p), kt0 + 1) == kTileAllFalse)
      p = w.step(p);
  }
  return p;
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

// Reduce-scatter over the warp: lane l returns the sum over all 32 lanes of
// their v[l] (recursive halving; the order of the additions is fixed).
// v is clobbered.
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// dK of key row j, shared by four threads: the thread of warp w (of the
// sixteen epilogue warps) holds head dims [32 cq, 32 cq + 32) (cq = w / 4) of
// the row in its TMEM lane (the dK' accumulator, the gradient of the rotated,
// normed row divided by the softmax scale). With x the raw k row,
// r = 1 / sqrt(mean x^2 + eps), g = scale dK', dy = R^T g (the rotation with
// sin negated) and g' = w dy:
//   dk = r g' - (r^3 / D) x (x . g'),   dW_k gathers dy x r.
// The raw row (bf16: the two 64-column halves of kOffK; fp32: four 32-column
// boxes over kOffK..kOffV) and the row's fp32 (cos, sin) (four 32-float boxes
// at kOffQ) were staged by TMA, 128B-swizzled. The two row sums (x.x, x.g')
// are completed through `ex_ss` and `ex_xg` in shared memory, between named
// barriers of the epilogue warps; sWk holds the k norm weights. A 16-bit dk
// row goes to `stage` (the operand-tile layout, stored by TMA afterwards); an
// fp32 one is stored directly. Returns, in lane l, the sum of dy x r at column
// 32 cq + l over the warp's 32 rows.
// Out of line: it runs once per CTA, and inlined it would spread the roles'
// hot loops over more instruction-cache lines.
template <bool QKT, bool F16>
__device__ __noinline__ float dk_quarter_rows(const BwdParams& P, const uint8_t* sm, uint32_t tacc, bool have, int b,
                                              int hk, int j, int r, int cq, bool key_ok, int lane, float* ex_ss,
                                              float* ex_xg, const float* sWk, uint8_t* stage) {
  const Common& c = P.c;
  // eight consecutive dims d0 .. d0 + 7 of the quarter (d0 a multiple of 8)
  auto load_x8 = [&](int d0, float (&x8)[8]) {
    if constexpr (QKT) {
      const uint4 u = *reinterpret_cast<const uint4*>(sm + kOffK + (cq >> 1) * kHalfBytes +
                                                      sw128_off(r, 4 * (cq & 1) + (d0 >> 3)));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x8[2 * e] = lo16<F16>(w[e]);
        x8[2 * e + 1] = hi16<F16>(w[e]);
      }
    } else {
      const uint8_t* box = sm + kOffK + cq * kBoxBytes;
      const float4 a = *reinterpret_cast<const float4*>(box + sw128_off(r, d0 >> 2));
      const float4 bq = *reinterpret_cast<const float4*>(box + sw128_off(r, (d0 >> 2) + 1));
      x8[0] = a.x; x8[1] = a.y; x8[2] = a.z; x8[3] = a.w; x8[4] = bq.x; x8[5] = bq.y; x8[6] = bq.z; x8[7] = bq.w;
    }
  };
  // (cos, sin) of the quarter's pairs 2t, 2t + 1 (pairs 16 cq + 2t ..)
  auto tab_chunk = [&](int t) -> float4 {
    return *reinterpret_cast<const float4*>(sm + kOffQ + cq * kBoxBytes + sw128_off(r, t));
  };
  float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
  for (int d0 = 0; d0 < 32; d0 += 8) {
    float x8[8];
    load_x8(d0, x8);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      ss0 = fmaf(x8[e], x8[e], ss0);
      ss1 = fmaf(x8[e + 1], x8[e + 1], ss1);
    }
  }
  ex_ss[cq * kTile + r] = ss0 + ss1;
  named_bar(kBarIdEpi, kEpiThreads);
  const float rr =
      rsqrtf((((ex_ss[r] + ex_ss[kTile + r]) + ex_ss[2 * kTile + r]) + ex_ss[3 * kTile + r]) * (1.0f / kD) + c.eps);
  const float sc = c.scale;
  const float4* w4 = reinterpret_cast<const float4*>(sWk + 32 * cq);
  // g' = w R^T (scale dK') of the quarter, kept for dk; u gathers dy x r for dW_k
  float gw[32], u[32];
  float xg = 0.f;
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {  // 16 dims per TMEM load
    uint32_t v[16];
    if (have) {
      tmem_ld16_issue(tacc + 16 * h2, v);
      tmem_ld_wait16(v);
    } else {
#pragma unroll
      for (int t = 0; t < 16; ++t) v[t] = 0u;
    }
#pragma unroll
    for (int c8 = 0; c8 < 2; ++c8) {
      const int d0 = 16 * h2 + 8 * c8;  // dims d0 .. d0 + 7 of the quarter: pairs d0/2 .. d0/2 + 3
      float x8[8];
      load_x8(d0, x8);
      const float4 t0 = tab_chunk(d0 >> 2), t1 = tab_chunk((d0 >> 2) + 1);
      const float cs[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      const float4 wa = w4[d0 >> 2], wb = w4[(d0 >> 2) + 1];
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = d0 + 2 * e, vi = 8 * c8 + 2 * e;
        const float g0 = __uint_as_float(v[vi]) * sc, g1 = __uint_as_float(v[vi + 1]) * sc;
        const float cc = cs[2 * e], sn = cs[2 * e + 1];
        const float dy0 = fmaf(g0, cc, g1 * sn), dy1 = fmaf(g1, cc, -g0 * sn);
        gw[t] = wv[2 * e] * dy0;
        gw[t + 1] = wv[2 * e + 1] * dy1;
        xg = fmaf(x8[2 * e], gw[t], fmaf(x8[2 * e + 1], gw[t + 1], xg));
        u[t] = key_ok ? dy0 * x8[2 * e] * rr : 0.f;
        u[t + 1] = key_ok ? dy1 * x8[2 * e + 1] * rr : 0.f;
      }
    }
  }
  const float colsum = warp_reduce_scatter32(u, lane);
  // x . g' over the whole row
  ex_xg[cq * kTile + r] = xg;
  named_bar(kBarIdEpi, kEpiThreads);
  xg = ((ex_xg[r] + ex_xg[kTile + r]) + ex_xg[2 * kTile + r]) + ex_xg[3 * kTile + r];
  const float c3 = rr * rr * rr * xg * (1.0f / kD);
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {  // dk = r g' - (r^3 / D) x (x . g')
    float x8[8];
    load_x8(8 * c8, x8);
#pragma unroll
    for (int e = 0; e < 8; ++e) u[8 * c8 + e] = fmaf(rr, gw[8 * c8 + e], -c3 * x8[e]);
  }
  {
    if constexpr (QKT) {
      // 16-bit dk: chunks 4 (cq % 2) .. + 3 of the row's half cq / 2 in the staging tile
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        *reinterpret_cast<uint4*>(stage + (cq >> 1) * kHalfBytes + sw128_off(r, 4 * (cq & 1) + c4)) =
            make_uint4(pack16<F16>(u[8 * c4], u[8 * c4 + 1]), pack16<F16>(u[8 * c4 + 2], u[8 * c4 + 3]),
                       pack16<F16>(u[8 * c4 + 4], u[8 * c4 + 5]), pack16<F16>(u[8 * c4 + 6], u[8 * c4 + 7]));
    } else if (key_ok) {
      store_chunk32(P.dk, b * P.dk_sb + (int64_t)j * P.dk_ss + hk * P.dk_sh, P.dk_dt, cq, u);
    }
  }
  return colsum;
}

// P^T of this thread's key against 32 queries iq0 .. iq0 + 31 of a chunk
// that needs masking (a bool tile with False elements, an additive mask
// broadcast over the queries, the causal diagonal, rows past S_q). Out of
// line: chunks without masking never run it, and inlined it would spread
// the compute warps' hot loop over more instruction-cache lines.
// It reads the warp's 32 S^T columns at TMEM address tS and writes P^T (16-bit
// pairs) over the first 16 of them itself, so that no array crosses the call.
template <int MK, bool CAUSAL, bool F16>
__device__ __noinline__ void p_masked(const Common& c, uint32_t tS, float key_term, int b, int h, int iq0, int j,
                                      bool key_ok, uint8_t flag, bool mask_bcast_q, const float* lse) {
  uint32_t sv[32], pw[16];
  tmem_ld32(tS, sv);
#pragma unroll
  for (int t2 = 0; t2 < 16; ++t2) {
    float p2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 2 * t2 + e;
      const float s2 = score2<MK, CAUSAL>(c, __uint_as_float(sv[t]), key_term, b, h, iq0 + t, j, key_ok, flag,
                                          mask_bcast_q);
      p2[e] = ex2(s2 - lse[t]);  // LSE = +inf for rows without keys or past S_q: P = 0
    }
    pw[t2] = pack16<F16>(p2[0], p2[1]);
  }
  tmem_st16(tS, pw);
  tmem_st_wait();
}

// ---- epilogue of the sixteen compute, drain and prologue warps, once their
// walks are over (n query tiles; `ok` is false after an abort). Warp w holds key
// rows 32 (w % 4) .. (its TMEM lanes) and head dims [32 cq, 32 cq + 32)
// (cq = w / 4) of dV and dK'. Once every MMA has completed, the K tile, the Q'
// ring and the dO ring are free: the raw k rows and the tile's fp32 (cos, sin)
// rows are staged by TMA (K tile, Q' ring) while dV is laid out in the dO ring
// and stored by TMA; then dk (inverse rotation + RMSNorm backward) is laid out
// in the dS buffers and stored by TMA (16-bit k; fp32 rows are stored
// directly), and each warp writes its partial sums of the k norm-weight
// gradient. The row sums are exchanged through the stat area and the second
// dO stage.
// Out of line, with every index derived again from the thread and block
// coordinates, so that nothing it needs stays live in registers through the
// main loops: with its values held across the loop (inlined, or called with
// them as arguments) the whole kernel took 12% longer at the 96-register cap
// (Flux1 1024px backward: 1039 us against 924 us).
template <bool QKT, bool F16>
__device__ __noinline__ void bwd_epilogue(const BwdParams& P, uint8_t* sm, int n, bool ok) {
  const Common& c = P.c;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  const uint32_t* tslot = reinterpret_cast<const uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(const_cast<uint32_t*>(tslot) + 1);
  const uint32_t tmem = *tslot;
  const long long budget = c.wait_budget;
  const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
  const int kt = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const bool phantom = kt >= c.nKt;
  const int qd = warp & 3, cq = warp >> 2;
  const int r = qd * 32 + lane_id;
  const int j = kt * kTile + r;
  const bool key_ok = j < c.Skv;
  const uint32_t lanebits = static_cast<uint32_t>(qd * 32) << 16;
  // the compute warps learn here that every MMA is done (the MMA thread's last
  // commit; the barrier below orders the rest)
  if (warp < kComputeWarps && ok && n > 0) ok = wait_bar_warp(&bars[kBarFinal], 0, abort_flag, budget);
  // one decision for the sixteen warps (they share named barriers below)
  if (!named_bar_any(kBarIdEpi, kEpiThreads, !ok) && !phantom) {
    tc_fence_after();
    float* ex_ss = reinterpret_cast<float*>(sm + kOffStat);  // the stats are consumed (2 KB)
    float* ex_xg = reinterpret_cast<float*>(sm + kOffDO + kQTileBytes);  // the second dO stage
    float* sWk = reinterpret_cast<float*>(sm + kOffW);       // k norm weights
    const int ty = P.k_s_first ? kt * kTile : hk, tz = P.k_s_first ? hk : kt * kTile;
    if (tid == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bars[kBarEpi], (QKT ? kTileBytes : 2 * kTileBytes) + 4 * kBoxBytes);
      if constexpr (QKT) {
        tma_load_4d(sm + kOffK, &P.tmap_k, &bars[kBarEpi], 0, ty, tz, b);
        tma_load_4d(sm + kOffK + kHalfBytes, &P.tmap_k, &bars[kBarEpi], 64, ty, tz, b);
      } else {
#pragma unroll
        for (int x = 0; x < 4; ++x)
          tma_load_4d(sm + kOffK + x * kBoxBytes, &P.tmap_k, &bars[kBarEpi], 32 * x, ty, tz, b);
      }
      const int trow = (c.tab_k_sb != 0 ? b * c.Skv : 0) + kt * kTile;
#pragma unroll
      for (int x = 0; x < 4; ++x) tma_load_2d(sm + kOffQ + x * kBoxBytes, &P.tmap_tab_k, &bars[kBarEpi], 32 * x, trow);
    }
    if (tid < kD) sWk[tid] = __ldg(c.wk + tid);
    {
      // dV: this thread's 32 columns of row r, 16-bit, into the dO ring in the
      // operand-tile layout
      uint8_t* stage = sm + kOffDO + (cq >> 1) * kHalfBytes;
      uint32_t v[32];
      if (n > 0) {
        tmem_ld32(tmem + 256 + lanebits + 32 * cq, v);
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) v[t] = 0u;
      }
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        *reinterpret_cast<uint4*>(stage + sw128_off(r, 4 * (cq & 1) + c4)) =
            make_uint4(pack16<F16>(__uint_as_float(v[8 * c4]), __uint_as_float(v[8 * c4 + 1])),
                       pack16<F16>(__uint_as_float(v[8 * c4 + 2]), __uint_as_float(v[8 * c4 + 3])),
                       pack16<F16>(__uint_as_float(v[8 * c4 + 4]), __uint_as_float(v[8 * c4 + 5])),
                       pack16<F16>(__uint_as_float(v[8 * c4 + 6]), __uint_as_float(v[8 * c4 + 7])));
      fence_proxy_async_smem();
    }
    if (!named_bar_any(kBarIdEpi, kEpiThreads, !wait_bar_warp(&bars[kBarEpi], 0, abort_flag, budget))) {
      if (tid == 0) {  // the staged dV rows (rows past S_kv are not written)
        const int vy = P.dv_s_first ? kt * kTile : hk, vz = P.dv_s_first ? hk : kt * kTile;
        tma_store_4d(&P.tmap_dv, sm + kOffDO, 0, vy, vz, b);
        tma_store_4d(&P.tmap_dv, sm + kOffDO + kHalfBytes, 64, vy, vz, b);
        bulk_commit_group();
      }
      const float colsum = dk_quarter_rows<QKT, F16>(P, sm, tmem + 384 + lanebits + 32 * cq, n > 0, b, hk, j, r,
                                                     cq, key_ok, lane_id, ex_ss, ex_xg, sWk, sm + kOffDS);
      // this warp's column sums over its 32 rows: one partial row per warp
      // quarter (rows 32 qd ..), added in a fixed order by the reduction
      P.dwk_part[((((int64_t)b * c.Hkv + hk) * c.nKt + kt) * 4 + qd) * kD + 32 * cq + lane_id] = colsum;
      if constexpr (QKT) {
        fence_proxy_async_smem();
        named_bar(kBarIdEpi, kEpiThreads);
        if (tid == 0) {
          const int ky = P.dk_s_first ? kt * kTile : hk, kz = P.dk_s_first ? hk : kt * kTile;
          tma_store_4d(&P.tmap_dk, sm + kOffDS, 0, ky, kz, b);
          tma_store_4d(&P.tmap_dk, sm + kOffDS + kHalfBytes, 64, ky, kz, b);
          bulk_commit_group();
        }
      }
      if (tid == 0) bulk_wait_read_all();  // the staged rows are read before the CTA may exit
    }
  }
}

// ELEM: the mask varies along the queries (per-element terms); a mask that is
// broadcast over the queries reduces to one term per key.
template <int MK, bool CAUSAL, bool QKT, bool ELEM, bool F16>
__device__ __forceinline__ void bwd_body(const BwdParams& P) {
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
  uint32_t* scratch = tslot + 2;  // [0]: sink for pin_loads; [1]: 1 when the K' tile came finished from the forward

  const Common& c = P.c;
  const int tid = threadIdx.x, warp = tid >> 5, lane_id = tid & 31;
  const int kt = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;  // key tile, K/V head, batch
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
    for (int s = 0; s < kDOStages; ++s) {
      mbar_init(&bars[kBarDOFull + s], 1);
      mbar_init(&bars[kBarDOFree + s], 1 + kDrainWarps);  // the dV MMAs, and the drain's box reads
    }
    mbar_init(&bars[kBarSFull], 1);
    mbar_init(&bars[kBarDPFull], 1);
    mbar_init(&bars[kBarPDone], kComputeWarps * 32);
    mbar_init(&bars[kBarCDone], kComputeWarps * 32);
    mbar_init(&bars[kBarDQ], 1);
    mbar_init(&bars[kBarBFree], kDrainWarps * 32);
    mbar_init(&bars[kBarFinal], 1);
    mbar_init(&bars[kBarEpi], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane_id == 0 && P.c.nQt > 0) {  // the maps exist only when there is work
    tma_prefetch_desc(&P.tmap_v);
    tma_prefetch_desc(&P.tmap_do);
    tma_prefetch_desc(&P.tmap_dq);
    tma_prefetch_desc(&P.tmap_k);
    tma_prefetch_desc(&P.tmap_tab_k);
    if (P.kp_ready) tma_prefetch_desc(&P.tmap_kc);
    tma_prefetch_desc(&P.tmap_q);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote copy or arrival
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t crank = cluster_rank();
  const long long budget = c.wait_budget;
  const bool phantom = kt >= c.nKt;  // pads the cluster when the key-tile count is odd
  QWalk W;
  W.begin = CAUSAL ? min(c.nQt, kt0) : 0;
  W.len = c.nQt - W.begin;
  W.rot = W.len > 0 ? static_cast<int>((static_cast<int64_t>(kt0 / 2) * W.len) / ((c.nKt + 1) / 2)) : 0;
  W.h0 = hk * c.group;
  W.group = c.group;
  int useful = 0;  // (query head, query tile) pairs this CTA's own key tile needed (compute warps)

  if (warp < kComputeWarps) {
    // ------------------------------------------------------------ compute
    const int qd = warp & 3, hq = warp >> 2;  // TMEM lane quarter, query half of a tile
    const int r = qd * 32 + lane_id;          // key row in the tile / TMEM lane
    const int j = kt * kTile + r;
    const bool key_ok = j < c.Skv;
    const uint32_t lanebits = static_cast<uint32_t>(qd * 32) << 16;
    // masks that do not depend on the query row: one term per key and head
    const bool mask_bcast_q = MK != kMaskNone && c.m_sq == 0;
    auto key_term_of = [&](int h) {
      float t = 0.f;
      if (mask_bcast_q && key_ok) {
        const int64_t off = b * c.m_sb + h * c.m_sh + j;
        if constexpr (MK == kMaskBool) t = __ldg(static_cast<const uint8_t*>(c.mask) + off) ? 0.f : -INFINITY;
        else if constexpr (MK == kMaskF32) t = __ldg(static_cast<const float*>(c.mask) + off) * kLog2e;
        else if constexpr (MK == kMaskBF16) t = __bfloat162float(static_cast<const __nv_bfloat16*>(c.mask)[off]) * kLog2e;
      }
      return key_ok ? t : -INFINITY;
    };
    int key_h = W.h0;
    float key_term = key_term_of(key_h);
    const float sc = c.scale_log2;
    const int qh0 = 64 * hq;  // this warp's first query of a tile
    bool ok = true;
    int n = 0;
    for (WPos m = next_pos<MK>(c, b, W, W.start(), kt0); ok && W.more(m);
         m = next_pos<MK>(c, b, W, W.step(m), kt0), ++n) {
      const int qt = W.qt(m), h = W.head(m);
      if (h != key_h) {
        key_h = h;
        key_term = key_term_of(h);
      }
      const uint8_t flag = own_flag<MK>(c, b, h, qt, kt);
      useful += (flag != kTileAllFalse && (!CAUSAL || qt >= kt)) ? 1 : 0;
      const int sq = n % kQStages;
      if (!(ok = wait_bar_warp(&bars[kBarSFull], n & 1, abort_flag, budget))) break;
      // the prologue's LSE/Delta for this stage become visible through this wait
      if (!(ok = wait_bar_warp(&bars[kBarQFull + sq], (n / kQStages) & 1, abort_flag, budget))) break;
      tc_fence_after();
      const float* st_lse = stat + sq * 2 * kTile;
      const float* st_dl = st_lse + kTile;
      // ---- P^T = exp2(S^T * scale*log2e - LSE*log2e), 16-bit into TMEM, per 32-query chunk;
      // kept in registers for dS^T as well, since S^T(n+1) overwrites X as soon
      // as the dV MMAs have read it
      uint32_t pwa[32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int q0 = qh0 + 32 * ch;  // the chunk's first query in the tile
        const int iq0 = qt * kTile + q0;
        const uint32_t tS = tmem + lanebits + kColX + q0;
        // plain chunks: every query row valid, no mask values, no causal diagonal
        const bool plain = flag != kTileAllFalse && iq0 + 32 <= c.Sq &&
                           (MK == kMaskNone || mask_bcast_q || (MK == kMaskBool && flag == kTileAllTrue)) &&
                           (!CAUSAL || iq0 >= kt * kTile + kTile - 1);
        uint32_t pw[16];
        if (!plain && !ELEM) {
          p_masked<MK, CAUSAL, F16>(c, tS, key_term, b, h, iq0, j, key_ok, flag, mask_bcast_q, st_lse + q0);
          tmem_ld16_issue(tS, pw);
          tmem_ld_wait16(pw);
        } else {
          uint32_t sv[32];
          tmem_ld32(tS, sv);
          if (plain) {
            const float2 sc2 = make_float2(sc, sc), kt2 = make_float2(key_term, key_term);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              const float4 l = *reinterpret_cast<const float4*>(st_lse + q0 + 4 * v4);
              const float2 c01 = __fadd2_rn(kt2, make_float2(-l.x, -l.y)), c23 = __fadd2_rn(kt2, make_float2(-l.z, -l.w));
              const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sv[4 * v4]), __uint_as_float(sv[4 * v4 + 1])), sc2, c01);
              const float2 x23 =
                  __ffma2_rn(make_float2(__uint_as_float(sv[4 * v4 + 2]), __uint_as_float(sv[4 * v4 + 3])), sc2, c23);
              pw[2 * v4] = pack16<F16>(ex2(x01.x), ex2(x01.y));
              pw[2 * v4 + 1] = pack16<F16>(ex2(x23.x), ex2(x23.y));
            }
          } else if constexpr (ELEM) {
            // per-element mask terms of the 32 queries, 16 at a time (loads pinned)
            const bool elem_mask = key_ok && flag != kTileAllFalse && !(MK == kMaskBool && flag == kTileAllTrue);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t raw[16];
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                raw[t] = 0u;
                const int iq = iq0 + 16 * hh + t;
                if (elem_mask && iq < c.Sq) {
                  const int64_t off = b * c.m_sb + h * c.m_sh + (int64_t)iq * c.m_sq + j;
                  if constexpr (MK == kMaskBool) raw[t] = __ldg(static_cast<const uint8_t*>(c.mask) + off) ? 0u : 1u;
                  else if constexpr (MK == kMaskF32)
                    raw[t] = __float_as_uint(ldg_nc_f32(static_cast<const float*>(c.mask) + off));
                  else raw[t] = static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(c.mask) + off)) << 16;
                }
              }
              uint32_t folded = 0;
#pragma unroll
              for (int t = 0; t < 16; ++t) folded ^= raw[t];
              pin_loads(folded, scratch);
#pragma unroll
              for (int t2 = 0; t2 < 8; ++t2) {
                float p2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int tl = 2 * t2 + e, t = 16 * hh + tl;
                  const float mterm = (MK == kMaskBool) ? (raw[tl] ? -INFINITY : 0.f) : __uint_as_float(raw[tl]) * kLog2e;
                  const float s2 = score2_term<CAUSAL>(c, __uint_as_float(sv[t]), key_term, mterm, iq0 + t, j, flag);
                  p2[e] = ex2(s2 - st_lse[q0 + t]);
                }
                pw[8 * hh + t2] = pack16<F16>(p2[0], p2[1]);
              }
            }
          }
          tmem_st16(tS, pw);  // the first 16 of the chunk's 32 S^T columns
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) pwa[16 * ch + i] = pw[i];
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kBarPDone]);
      // ---- dS^T = P^T (dP^T - Delta), 16-bit into shared memory (row r, K-major)
      // (dS^T(n-1) is consumed: its MMAs completed before dP^T(n) did)
      if (!(ok = wait_bar_warp(&bars[kBarDPFull], n & 1, abort_flag, budget))) break;
      tc_fence_after();
      {
        // 16 queries at a time; each TMEM load is issued before the previous
        // block is processed
        uint32_t da[16], db[16];
        uint8_t* dsb = sm + kOffDS + hq * kHalfBytes;
        tmem_ld16_issue(tmem + lanebits + kColY + qh0, da);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t(&cur)[16] = (k & 1) ? db : da;
          uint32_t(&nxt)[16] = (k & 1) ? da : db;
          tmem_ld_wait16(cur);
          if (k < 3) tmem_ld16_issue(tmem + lanebits + kColY + qh0 + 16 * (k + 1), nxt);
          const int q0 = qh0 + 16 * k;
#pragma unroll
          for (int u = 0; u < 2; ++u) {  // 8 queries = one 16-byte chunk of the dS^T row
            const float4 d0 = *reinterpret_cast<const float4*>(st_dl + q0 + 8 * u);
            const float4 d1 = *reinterpret_cast<const float4*>(st_dl + q0 + 8 * u + 4);
            const float2 ndl[4] = {make_float2(-d0.x, -d0.y), make_float2(-d0.z, -d0.w), make_float2(-d1.x, -d1.y),
                                   make_float2(-d1.z, -d1.w)};
            uint32_t out[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t pp = pwa[8 * k + 4 * u + e];
              const float2 dp = make_float2(__uint_as_float(cur[8 * u + 2 * e]), __uint_as_float(cur[8 * u + 2 * e + 1]));
              const float2 ds = __fmul2_rn(make_float2(lo16<F16>(pp), hi16<F16>(pp)), __fadd2_rn(dp, ndl[e]));
              out[e] = pack16<F16>(ds.x, ds.y);
            }
            *reinterpret_cast<uint4*>(dsb + sw128_off(r, 2 * k + u)) = make_uint4(out[0], out[1], out[2], out[3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[kBarCDone]);
    }
    bwd_epilogue<QKT, F16>(P, sm, n, ok);
  } else if (warp < kWarpDrain0 + kDrainWarps) {
    // ------------------------------------------------------------ dQ drain
    // A tile's dQ'^T (128 head dims x 128 queries, fp32) leaves TMEM in two
    // 64-query halves (64 registers per thread); the columns are released once
    // both are read. Warp qd stages head dims [32 qd, +32) of a half as a
    // [64 query][32] box in the tile's dO stage (idle once the dV MMAs are
    // done; the dO loads refill it only after kBarDOFree has the drain's
    // arrivals as well) and lane 0 adds the box into the global accumulator
    // (TMA bulk reduce); the second half reuses the box once the first reduce
    // has read it. Nothing on the tensor core's path waits for these copies,
    // and the warps never wait for one another.
    const int qd = warp & 3;
    const uint32_t lanebits = static_cast<uint32_t>(qd * 32) << 16;
    const float scale = c.scale;
    const bool leader = lane_id == 0;
    const uint32_t chunk = static_cast<uint32_t>(lane_id) >> 2, word = (lane_id & 3) * 4;
    int n = 0;
    bool ok = true;
    for (WPos m = next_pos<MK>(c, b, W, W.start(), kt0); ok && W.more(m);
         m = next_pos<MK>(c, b, W, W.step(m), kt0), ++n) {
      const int qt = W.qt(m), h = W.head(m);
      const int sd = n % kDOStages;
      uint8_t* box = sm + kOffDO + sd * kQTileBytes + qd * kRBoxBytes;
      if (!(ok = wait_bar_warp(&bars[kBarDQ], n & 1, abort_flag, budget))) break;
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lanebits + kColY + kDrainRows * half, v0);
        tmem_ld32(tmem + lanebits + kColY + kDrainRows * half + 32, v1);
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(&bars[kBarBFree]);
          if (leader) bulk_wait_read_all();  // the first half's reduce has read the box
          __syncwarp();
        }
#pragma unroll
        for (int q = 0; q < kDrainRows; ++q) {  // row q of the box: 32 consecutive head dims, 128B-swizzled
          const uint32_t v = q < 32 ? v0[q] : v1[q - 32];
          *reinterpret_cast<float*>(box + q * 128 + ((chunk ^ (q & 7)) << 4) + word) = __uint_as_float(v) * scale;
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int row = qt * kTile + kDrainRows * half;
        if (leader && row < c.Sq) {  // a half wholly past S_q adds nothing
          tma_reduce_add_4d(&P.tmap_dq, box, 32 * qd, h, row, b);
          bulk_commit_group();
        }
      }
      if (leader) {
        bulk_wait_read_all();  // the second half's reduce has read the box
        mbar_arrive(&bars[kBarDOFree + sd]);
      }
    }
    if (leader) bulk_wait_all();  // the reduces are complete before the epilogue reuses the buffer
    bwd_epilogue<QKT, F16>(P, sm, n, ok);
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
      // the tile's rows have landed: raw 16-bit rows, or the K' tile that the
      // forward published (then nothing is left to do); fp32 rows are read
      // from global memory below
      ok = wait_bar(&bars[kBarKRaw], 0, abort_flag, budget);
      const bool cached = *reinterpret_cast<volatile uint32_t*>(scratch + 1) != 0u;
      if constexpr (QKT) {
        for (int row = p; ok && !cached && row < kTile; row += kProlThreads) {
          const int jj = kt * kTile + row;
          if (jj < c.Skv)  // rows past S_kv stay TMA zeros
            rope_norm_inplace<F16>(sm + kOffK, row, c.wk, c.eps, c.tab16_k + b * c.tab_k_sb + (int64_t)jj * kPairs);
        }
      } else if (__all_sync(0xffffffffu, ok) && !cached) {
        // fp32 rows from global memory, four lanes per row, as the forward
        // builds them (every lane of the warp in every pass)
#pragma unroll 1
        for (int pass = 0; pass < kTile * 4 / kProlThreads; ++pass) {
          const int row = pass * (kProlThreads / 4) + (p >> 2), jj = kt * kTile + row;
          const bool valid = jj < c.Skv;
          const int jv = valid ? jj : 0;
          rope_norm_global_quad<F16>(c.k.p, b * c.k.sb + (int64_t)jv * c.k.ss + hk * c.k.sh, c.k.dt, c.wk, c.eps,
                                     c.tab_k + b * c.tab_k_sb + (int64_t)jv * kPairs, sm + kOffK, row, p & 3, valid,
                                     kHalfBytes);
        }
      }
    }
    if (ok) {
      fence_proxy_async_smem();
      mbar_arrive(&bars[kBarKFull]);
    }
    // the same decision in every prologue thread: a flag read after a plain
    // barrier could differ between threads if another role aborts meanwhile,
    // and the loop below has named barriers of its own
    ok = !named_bar_any(3, kProlThreads, *abort_flag != 0);
    // Q' rows arrive by TMA from the workspace (the forward's normalised,
    // rotated q rows); these threads stage each tile's LSE (base 2; +inf for
    // rows without keys or past S_q, so that P = 0) and Delta, loaded one tile
    // ahead. A stage's values are rewritten once both CTAs' MMAs have released
    // the stage (the compute warps have read them by then).
    float lse_c = -INFINITY, dl_c = 0.f;
    auto load_stats = [&](int iq0, int h) {
      lse_c = -INFINITY;
      dl_c = 0.f;
      if (iq0 + p < c.Sq) {
        const int64_t ri = ((int64_t)b * c.H + h) * c.Sq + iq0 + p;
        lse_c = ldg_nc_f32(P.lse + ri);
        dl_c = ldg_nc_f32(P.delta + ri);
      }
    };
    // A mask that varies along the queries: the mask rows of a tile (this
    // CTA's keys, the tile's 128 queries, one row per thread) are prefetched
    // into L2 a tile ahead of the compute warps, whose loads of them are
    // otherwise the backward's bottleneck.
    auto prefetch_mask = [&](int qt, int h) {
      if constexpr (ELEM) {
        constexpr int es = MK == kMaskF32 ? 4 : (MK == kMaskBF16 ? 2 : 1);
        const int iq = qt * kTile + p, j0 = kt * kTile;
        if (iq < c.Sq && j0 < c.Skv) {
          const uint8_t* row = static_cast<const uint8_t*>(c.mask) +
                               ((int64_t)b * c.m_sb + (int64_t)h * c.m_sh + (int64_t)iq * c.m_sq + j0) * es;
          const int nbytes = min(kTile, c.Skv - j0) * es;
          for (int off = 0; off < nbytes; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
        }
      }
    };
    WPos m = next_pos<MK>(c, b, W, W.start(), kt0);
    if (W.more(m)) {
      load_stats(W.qt(m) * kTile, W.head(m));
      prefetch_mask(W.qt(m), W.head(m));
    }
    int n = 0;
    for (; ok && W.more(m); ++n) {
      const WPos m_next = next_pos<MK>(c, b, W, W.step(m), kt0);
      const int sq = n % kQStages;
      const float l2 = (lse_c == -INFINITY) ? INFINITY : lse_c * kLog2e, dl = dl_c;
      if (n >= kQStages &&
          !(ok = wait_bar_cluster_warp(&bars[kBarQFree + sq], ((n / kQStages) - 1) & 1, abort_flag, budget)))
        break;
      stat[sq * 2 * kTile + p] = l2;
      stat[sq * 2 * kTile + kTile + p] = dl;
      if (W.more(m_next)) {
        load_stats(W.qt(m_next) * kTile, W.head(m_next));
        prefetch_mask(W.qt(m_next), W.head(m_next));
      }
      mbar_arrive(&bars[kBarQFull + sq]);
      m = m_next;
    }
    bwd_epilogue<QKT, F16>(P, sm, n, ok);
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA: raw K, V, raw Q
    if (lane_id == 0) {
      if (!phantom) {
        // K' as the forward published it (rows past S_kv read as zeros), else
        // the raw rows (16-bit), else a plain arrival (fp32 rows)
        const bool cached = P.kp_ready && P.kflags[((int64_t)b * c.Hkv + hk) * c.nKt + kt] != 0u;
        scratch[1] = cached ? 1u : 0u;
        if (cached) {
          mbar_arrive_expect_tx(&bars[kBarKRaw], kTileBytes);
          tma_load_4d(sm + kOffK, &P.tmap_kc, &bars[kBarKRaw], 0, hk, kt * kTile, b);
          tma_load_4d(sm + kOffK + kHalfBytes, &P.tmap_kc, &bars[kBarKRaw], 64, hk, kt * kTile, b);
        } else if constexpr (QKT) {
          const int y = P.k_s_first ? kt * kTile : hk, z = P.k_s_first ? hk : kt * kTile;
          mbar_arrive_expect_tx(&bars[kBarKRaw], kTileBytes);
          tma_load_4d(sm + kOffK, &P.tmap_k, &bars[kBarKRaw], 0, y, z, b);
          tma_load_4d(sm + kOffK + kHalfBytes, &P.tmap_k, &bars[kBarKRaw], 64, y, z, b);
        } else {
          mbar_arrive(&bars[kBarKRaw]);
        }
        const int vy = P.v_s_first ? kt * kTile : hk, vz = P.v_s_first ? hk : kt * kTile;
        mbar_arrive_expect_tx(&bars[kBarVFull], kTileBytes);
        tma_load_4d(sm + kOffV, &P.tmap_v, &bars[kBarVFull], 0, vy, vz, b);
        tma_load_4d(sm + kOffV + kHalfBytes, &P.tmap_v, &bars[kBarVFull], 64, vy, vz, b);
      } else {
        mbar_arrive(&bars[kBarVFull]);  // V is zeroed by the prologue, before K' is declared ready
      }
      int n = 0, q_issued = 0;
      for (WPos m = next_pos<MK>(c, b, W, W.start(), kt0); W.more(m); m = next_pos<MK>(c, b, W, W.step(m), kt0), ++n) {
        const int qt = W.qt(m), h = W.head(m);
        // this CTA's 64 Q' rows of the tile, into both CTAs' stage; the stage
        // holds the peer's 64 rows as well once kQTileBytes have landed
        const int sq = n % kQStages;
        if (n >= kQStages && !wait_bar_cluster(&bars[kBarQFree + sq], ((n / kQStages) - 1) & 1, abort_flag, budget))
          break;
        uint8_t* qrows = sm + kOffQ + sq * kQTileBytes + kPeerRowsBytes * crank;
        const int row = qt * kTile + kPeerRows * static_cast<int>(crank);
        mbar_arrive_expect_tx(&bars[kBarQRaw + sq], kQTileBytes);
        tma_load_4d_mc(qrows, &P.tmap_q, &bars[kBarQRaw + sq], 0, h, row, b, 0x3);
        tma_load_4d_mc(qrows + kHalfBytes, &P.tmap_q, &bars[kBarQRaw + sq], 64, h, row, b, 0x3);
        ++q_issued;
      }
      // drain: every issued load lands before the CTA exits (these waits do not
      // give up on abort; each is bounded)
      if (!phantom) {
        mbar_wait(&bars[kBarVFull], 0, budget);
        mbar_wait(&bars[kBarKRaw], 0, budget);
      }
      for (int x = max(0, q_issued - kQStages); x < q_issued; ++x)
        mbar_wait(&bars[kBarQRaw + x % kQStages], (x / kQStages) & 1, budget);
    }
  } else if (warp == kWarpTmaDO) {
    // ------------------------------------------------------------ TMA: dO
    if (lane_id == 0) {
      int n = 0, do_issued = 0;
      for (WPos m = next_pos<MK>(c, b, W, W.start(), kt0); W.more(m); m = next_pos<MK>(c, b, W, W.step(m), kt0), ++n) {
        const int qt = W.qt(m), h = W.head(m);
        const int sd = n % kDOStages;
        if (n >= kDOStages && !wait_bar(&bars[kBarDOFree + sd], ((n / kDOStages) - 1) & 1, abort_flag, budget)) break;
        const int row = qt * kTile;
        const int y = P.do_s_first ? row : h, z = P.do_s_first ? h : row;
        uint8_t* dst = sm + kOffDO + sd * kQTileBytes;
        mbar_arrive_expect_tx(&bars[kBarDOFull + sd], kQTileBytes);
        tma_load_4d(dst, &P.tmap_do, &bars[kBarDOFull + sd], 0, y, z, b);
        tma_load_4d(dst + kHalfBytes, &P.tmap_do, &bars[kBarDOFull + sd], 64, y, z, b);
        ++do_issued;
      }
      for (int x = max(0, do_issued - kDOStages); x < do_issued; ++x)
        mbar_wait(&bars[kBarDOFull + x % kDOStages], (x / kDOStages) & 1, budget);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue
    if (lane_id == 0) {
      constexpr uint32_t idesc_sdp = idesc16(F16, 128, 128, 0, 0);  // S^T, dP^T: N = 128 queries
      constexpr uint32_t idesc_kv = idesc16(F16, 128, 128, 0, 1);   // dV, dK': N = 128 head dims
      constexpr uint32_t idesc_q = idesc16(F16, 128, 128, 1, 1);    // dQ'^T = K'^T dS^T
      const uint64_t dKk = sdesc_sw128(smem_u32(sm + kOffK), 16, 1024);
      const uint64_t dKm = sdesc_sw128(smem_u32(sm + kOffK), kHalfBytes, 1024);
      const uint64_t dVk = sdesc_sw128(smem_u32(sm + kOffV), 16, 1024);
      const uint64_t dQk0 = sdesc_sw128(smem_u32(sm + kOffQ), 16, 1024);
      const uint64_t dQm0 = sdesc_sw128(smem_u32(sm + kOffQ), kHalfBytes, 1024);
      const uint64_t dOk0 = sdesc_sw128(smem_u32(sm + kOffDO), 16, 1024);
      const uint64_t dOm0 = sdesc_sw128(smem_u32(sm + kOffDO), kHalfBytes, 1024);
      const uint64_t dSk = sdesc_sw128(smem_u32(sm + kOffDS), 16, 1024);
      const uint64_t dSm = sdesc_sw128(smem_u32(sm + kOffDS), kHalfBytes, 1024);
      const uint32_t tX = tmem + kColX, tY = tmem + kColY, tdV = tmem + kColDV, tdK = tmem + kColDK;
      int ntiles = W.len * W.group;  // query tiles in the walk (bool masks skip the tiles both key tiles mask out)
      if constexpr (MK == kMaskBool) {
        ntiles = 0;
        for (WPos m = next_pos<MK>(c, b, W, W.start(), kt0); W.more(m); m = next_pos<MK>(c, b, W, W.step(m), kt0)) ++ntiles;
      }
      auto issue_s = [&](int n) -> bool {  // S^T(n) into X
        const int sq = n % kQStages;
        if (!wait_bar(&bars[kBarQRaw + sq], (n / kQStages) & 1, abort_flag, budget)) return false;
        tc_fence_after();
        const uint64_t dQk = sdesc_add(dQk0, sq * kQTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tX, sdesc_add(dKk, kofs128(kk)), sdesc_add(dQk, kofs128(kk)), idesc_sdp, kk > 0);
        mma_commit(&bars[kBarSFull]);
        return true;
      };
      auto issue_dp = [&](int n) -> bool {  // dP^T(n) into Y
        const int sd = n % kDOStages;
        if (!wait_bar(&bars[kBarDOFull + sd], (n / kDOStages) & 1, abort_flag, budget)) return false;
        tc_fence_after();
        const uint64_t dOk = sdesc_add(dOk0, sd * kQTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tY, sdesc_add(dVk, kofs128(kk)), sdesc_add(dOk, kofs128(kk)), idesc_sdp, kk > 0);
        mma_commit(&bars[kBarDPFull]);
        return true;
      };
      bool ok = wait_bar(&bars[kBarKFull], 0, abort_flag, budget) && wait_bar(&bars[kBarVFull], 0, abort_flag, budget);
      bool issued = false;
      if (ok && ntiles > 0) {
        issued = true;
        ok = issue_s(0) && issue_dp(0);
      }
      for (int n = 0; ok && n < ntiles; ++n) {
        const int sq = n % kQStages, sd = n % kDOStages;
        // dV += P^T dO: P^T (16-bit) in X, read from TMEM
        if (!(ok = wait_bar(&bars[kBarPDone], n & 1, abort_flag, budget))) break;
        tc_fence_after();
        const uint64_t dOm = sdesc_add(dOm0, sd * kQTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tdV, tX + p_col(kk), sdesc_add(dOm, mofs(kk)), idesc_kv, (n > 0 || kk > 0));
        mma_commit(&bars[kBarDOFree + sd]);
        // S^T(n+1) over P^T(n) (the dV MMAs above read it first: same issuing
        // thread, in order), so that the compute warps find it when they are
        // done with dS^T(n)
        if (n + 1 < ntiles && !(ok = issue_s(n + 1))) break;
        if (!(ok = wait_bar(&bars[kBarCDone], n & 1, abort_flag, budget))) break;
        tc_fence_after();
        // dQ'^T = K'^T dS^T over dP^T (read by the compute warps before they
        // signalled); first, so that the drain starts early
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tY, sdesc_add(dKm, mofs(kk)), sdesc_add(dSm, mofs(kk)), idesc_q, kk > 0);
        mma_commit(&bars[kBarDQ]);
        // dK' += dS^T Q'
        const uint64_t dQm = sdesc_add(dQm0, sq * kQTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tdK, sdesc_add(dSk, kofs128(kk)), sdesc_add(dQm, mofs(kk)), idesc_kv, (n > 0 || kk > 0));
        mma_commit_mc(&bars[kBarQFree + sq], 0x3);  // the Q' stage is released in both CTAs' view
        // dP^T(n+1) over dQ'^T(n) once the drain has read it
        if (n + 1 < ntiles) {
          if (!(ok = wait_bar(&bars[kBarBFree], n & 1, abort_flag, budget))) break;
          ok = issue_dp(n + 1);
        }
      }
      if (issued) {
        // every issued MMA done: the epilogue reads dV and dK' (on abort: before TMEM is released)
        mma_commit(&bars[kBarFinal]);
        if (!ok) mbar_wait(&bars[kBarFinal], 0, budget);
      }
    }
  }

  // ---- tile counters
  // the lanes of the single-thread roles wait for their lane 0 here, at a warp
  // barrier, rather than at the block barrier below
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (!*abort_flag) {
    if (!phantom && tid == 0) {
      atomicAdd(c.counters + kCtrTilesSkipped, (unsigned long long)(c.group * c.nQt - useful));
      atomicAdd(c.counters + kCtrTilesTotal, (unsigned long long)(c.group * c.nQt));
    }
  } else if (tid == 0) {
    record_timeout(c);
  }
  tc_fence_before();
  cluster_sync();  // no DSMEM copy or remote arrival may target a CTA that has exited
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

template <int MK, bool CAUSAL, bool QKT, bool ELEM, bool F16>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ BwdParams P) {
  grid_dependency_wait();
  if constexpr (MK == kMaskBool) {
    // A bool mask whose every element is True (found by the classify kernel
    // of this call or of the forward whose tables it reuses) masks nothing:
    // the unmasked body computes the same results without the per-tile class
    // lookups in every role's walk.
    if (*P.c.mask_any_false == 0u) {
      bwd_body<kMaskNone, CAUSAL, QKT, false, F16>(P);
      return;
    }
  }
  bwd_body<MK, CAUSAL, QKT, ELEM, F16>(P);
}

}  // namespace

template <int MK, bool CAUSAL, bool QKT, bool ELEM, bool F16>
cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  auto kern = bwd_kernel<MK, CAUSAL, QKT, ELEM, F16>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = opt_in_smem(kern, kBwdSmem, configured);
  if (e != cudaSuccess) return e;
  dim3 grid((p.c.nKt + kCluster - 1) / kCluster * kCluster, p.c.Hkv, p.c.B);  // whole clusters
  return launch_chained(kern, grid, dim3(kBwdThreads), kBwdSmem, stream, p);
}

template <bool QKT, bool F16>
cudaError_t launch_bwd_q(const BwdParams& p, cudaStream_t stream) {
  if (p.c.causal) return launch_bwd_t<kMaskNone, true, QKT, false, F16>(p, stream);  // masks and causal never combine
  const bool elem = p.c.m_sq != 0;  // the mask varies along the queries
  switch (p.c.mask_kind) {
    case kMaskBool:
      return elem ? launch_bwd_t<kMaskBool, false, QKT, true, F16>(p, stream)
                  : launch_bwd_t<kMaskBool, false, QKT, false, F16>(p, stream);
    case kMaskF32:
      return elem ? launch_bwd_t<kMaskF32, false, QKT, true, F16>(p, stream)
                  : launch_bwd_t<kMaskF32, false, QKT, false, F16>(p, stream);
    case kMaskBF16:
      return elem ? launch_bwd_t<kMaskBF16, false, QKT, true, F16>(p, stream)
                  : launch_bwd_t<kMaskBF16, false, QKT, false, F16>(p, stream);
    default: return launch_bwd_t<kMaskNone, false, QKT, false, F16>(p, stream);
  }
}

// Kernels are specialised on the mask kind, causal masking, whether q/k are
// staged by TMA, whether the mask varies along the queries and the 16-bit
// operand type, so that each carries only its own code. This translation
// unit holds one operand type (ST_OPERAND_F16).
#if ST_OPERAND_F16
cudaError_t launch_bwd_f16(const BwdParams& p, cudaStream_t stream) {
#else
cudaError_t launch_bwd_bf16(const BwdParams& p, cudaStream_t stream) {
#endif
  return p.qk_tma ? launch_bwd_q<true, ST_OPERAND_F16>(p, stream) : launch_bwd_q<false, ST_OPERAND_F16>(p, stream);
}

}  // namespace st
