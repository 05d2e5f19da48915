// Operand prologues: RMSNorm (fp32) + interleaved-pair RoPE of q or k rows,
// rounded to the 16-bit MMA operand type (bf16, or fp16 with F16) and written
// as K-major, 128B-swizzled UMMA operand tiles. The in-place forms work on raw
// rows that TMA has already landed in the operand layout (raw rows of the
// operand type); the global forms read bf16, fp16 or fp32 rows from global
// memory.
#pragma once
#include "st_common.cuh"

namespace st {

// Thread-per-row prologue on a tile that TMA has already filled with the raw
// bf16 rows (128B-swizzled, the operand layout): the thread reads its row,
// normalises and rotates it, and writes the bf16 result back in place. The
// swizzle makes eight consecutive rows hit eight different bank groups, so
// the 16-byte accesses are conflict-free. tab16: the row's 64 (cos, sin) in
// fp16 (16 loads of 16 bytes, all issued before the arithmetic); w: the norm
// weights in shared memory.
template <bool F16>
struct RowInplace {
  uint4 cs[kD / 8];  // (cos, sin) of pairs 4c .. 4c+3, fp16
  // Issues the row's table loads; finish() consumes them.
  __device__ __forceinline__ void prefetch(const __half2* __restrict__ tab16) {
    const uint4* t16 = reinterpret_cast<const uint4*>(tab16);
#pragma unroll
    for (int c = 0; c < kD / 8; ++c) cs[c] = ldg_nc_v4(t16 + c);
  }
  // The sum of squares is taken per 64-column half (even and odd columns
  // apart) and the halves added, the order of HalfRowPrologue, so that a K'
  // row built here equals the forward's bit for bit.
  __device__ __forceinline__ void finish(uint8_t* tile, int row, const float* w, float eps) const {
    float half_ss[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + hh * kHalfBytes + sw128_off(row, c));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = lo16<F16>(u[e]), hi = hi16<F16>(u[e]);
          a0 = fmaf(lo, lo, a0);
          a1 = fmaf(hi, hi, a1);
        }
      }
      half_ss[hh] = a0 + a1;
    }
    const float r = rsqrtf((half_ss[0] + half_ss[1]) * (1.0f / kD) + eps);
    const float4* w4 = reinterpret_cast<const float4*>(w);
#pragma unroll
    for (int c = 0; c < kD / 8; ++c) {
      uint4* p16 = reinterpret_cast<uint4*>(tile + (c >> 3) * kHalfBytes + sw128_off(row, c & 7));
      const uint4 v = *p16;
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      const uint32_t t[4] = {cs[c].x, cs[c].y, cs[c].z, cs[c].w};
      const float4 wa = w4[2 * c], wb = w4[2 * c + 1];
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      uint32_t out[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // pair 4c + e
        const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&t[e]));  // (cos, sin)
        const float n0 = lo16<F16>(u[e]) * wv[2 * e] * r, n1 = hi16<F16>(u[e]) * wv[2 * e + 1] * r;
        out[e] = pack16<F16>(n0 * sc.x - n1 * sc.y, n0 * sc.y + n1 * sc.x);
      }
      *p16 = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
};

template <bool F16>
__device__ __forceinline__ void rope_norm_inplace(uint8_t* tile, int row, const float* w, float eps,
                                                  const __half2* __restrict__ tab16) {
  RowInplace<F16> rp;
  rp.prefetch(tab16);
  rp.finish(tile, row, w, eps);
}

// Eight-lanes-per-row variant: lane part q = lane >> 2 (0..7) of row slot
// lane & 3 owns the 16-byte chunk q of both 64-column halves (head dims
// 8q..8q+7 and 64+8q..64+8q+7, pairs 4q.. and 32+4q..). The (cos, sin) loads of
// one instruction then cover four rows x 128 contiguous bytes (four cache
// lines) instead of one line per lane, and the swizzled tile accesses of four
// consecutive rows are conflict-free. The row's sum of squares is reduced
// over the eight lanes with shuffles, so all 32 lanes call finish().
template <bool F16>
struct OctRow {
  uint4 cs0, cs1;  // (cos, sin) fp16 of this lane's pairs in half 0 and half 1
  // Folds the loaded words into `acc`: a use that the compiler cannot move the
  // loads past (see pin_loads).
  __device__ __forceinline__ uint32_t fold(uint32_t acc) const {
    return acc ^ cs0.x ^ cs0.y ^ cs0.z ^ cs0.w ^ cs1.x ^ cs1.y ^ cs1.z ^ cs1.w;
  }
  __device__ __forceinline__ void prefetch(const __half2* __restrict__ tab16_row, int part) {
    const uint4* t = reinterpret_cast<const uint4*>(tab16_row);
    cs0 = ldg_nc_v4(t + part);
    cs1 = ldg_nc_v4(t + 8 + part);
  }
  __device__ __forceinline__ static void rotate8(uint4& v, const uint4& cs, const float* w8, float r) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    const uint32_t t[4] = {cs.x, cs.y, cs.z, cs.w};
    const float4 wa = *reinterpret_cast<const float4*>(w8), wb = *reinterpret_cast<const float4*>(w8 + 4);
    const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&t[e]));  // (cos, sin)
      const float n0 = lo16<F16>(u[e]) * wv[2 * e] * r, n1 = hi16<F16>(u[e]) * wv[2 * e + 1] * r;
      out[e] = pack16<F16>(n0 * sc.x - n1 * sc.y, n0 * sc.y + n1 * sc.x);
    }
    v = make_uint4(out[0], out[1], out[2], out[3]);
  }
  // Two rows at once (independent chains interleaved for instruction-level
  // parallelism); same contract as finish().
  // half: byte distance of the two 64-column halves (kHalfBytes for a
  // 128-row tile, half that for a 64-row one)
  __device__ __forceinline__ static void finish2(const OctRow& ra, const OctRow& rb, uint8_t* tile, int row_a,
                                                 int row_b, int part, const float* w, float eps, bool valid_a,
                                                 bool valid_b, uint32_t half = kHalfBytes) {
    uint4* pa0 = reinterpret_cast<uint4*>(tile + sw128_off(row_a, part));
    uint4* pa1 = reinterpret_cast<uint4*>(tile + half + sw128_off(row_a, part));
    uint4* pb0 = reinterpret_cast<uint4*>(tile + sw128_off(row_b, part));
    uint4* pb1 = reinterpret_cast<uint4*>(tile + half + sw128_off(row_b, part));
    uint4 va0 = *pa0, va1 = *pa1, vb0 = *pb0, vb1 = *pb1;
    const uint32_t ua[8] = {va0.x, va0.y, va0.z, va0.w, va1.x, va1.y, va1.z, va1.w};
    const uint32_t ub[8] = {vb0.x, vb0.y, vb0.z, vb0.w, vb1.x, vb1.y, vb1.z, vb1.w};
    float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 xa = make_float2(lo16<F16>(ua[e]), hi16<F16>(ua[e]));
      const float2 xb = make_float2(lo16<F16>(ub[e]), hi16<F16>(ub[e]));
      sa = __ffma2_rn(xa, xa, sa);
      sb = __ffma2_rn(xb, xb, sb);
    }
    float ssa = sa.x + sa.y, ssb = sb.x + sb.y;
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      ssa += __shfl_xor_sync(0xffffffffu, ssa, o);
      ssb += __shfl_xor_sync(0xffffffffu, ssb, o);
    }
    const float r_a = rsqrtf(ssa * (1.0f / kD) + eps), r_b = rsqrtf(ssb * (1.0f / kD) + eps);
    if (valid_a) {
      rotate8(va0, ra.cs0, w + 8 * part, r_a);
      rotate8(va1, ra.cs1, w + 64 + 8 * part, r_a);
    }
    if (valid_b) {
      rotate8(vb0, rb.cs0, w + 8 * part, r_b);
      rotate8(vb1, rb.cs1, w + 64 + 8 * part, r_b);
    }
    if (valid_a) {
      *pa0 = va0;
      *pa1 = va1;
    }
    if (valid_b) {
      *pb0 = vb0;
      *pb1 = vb1;
    }
  }
  // valid: the row exists (the eight lanes of the row agree); w: all 128 weights
  __device__ __forceinline__ void finish(uint8_t* tile, int row, int part, const float* w, float eps,
                                         bool valid) const {
    uint4* p0 = reinterpret_cast<uint4*>(tile + sw128_off(row, part));
    uint4* p1 = reinterpret_cast<uint4*>(tile + kHalfBytes + sw128_off(row, part));
    uint4 v0 = *p0, v1 = *p1;
    float a0 = 0.f, a1 = 0.f;
    const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float lo = lo16<F16>(u[e]), hi = hi16<F16>(u[e]);
      a0 = fmaf(lo, lo, a0);
      a1 = fmaf(hi, hi, a1);
    }
    float ss = a0 + a1;
    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
    ss += __shfl_xor_sync(0xffffffffu, ss, 8);
    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
    if (!valid) return;
    const float r = rsqrtf(ss * (1.0f / kD) + eps);
    rotate8(v0, cs0, w + 8 * part, r);
    rotate8(v1, cs1, w + 64 + 8 * part, r);
    *p0 = v0;
    *p1 = v1;
  }
};

// Half-row variant: two lanes of a warp (l and l ^ 16) share one row; lane
// half `hh` owns head dims [64*hh, 64*hh + 64) = the 64-column half `hh` of the
// swizzled tile. The (cos, sin) loads are issued by prefetch() before the raw
// rows are known to have landed; finish() waits for nothing itself.
template <bool F16>
struct HalfRowPrologue {
  uint4 cs[4];  // (cos, sin) fp16 of this lane's 32 pairs
  __device__ __forceinline__ void prefetch(const __half2* __restrict__ tab16_row, int hh) {
    const uint4* t16 = reinterpret_cast<const uint4*>(tab16_row) + 8 * hh;
#pragma unroll
    for (int c = 0; c < 4; ++c) cs[c] = ldg_nc_v4(t16 + c);
  }
  __device__ __forceinline__ void prefetch2(const __half2* __restrict__ tab16_row, int hh) {
    const uint4* t16 = reinterpret_cast<const uint4*>(tab16_row) + 8 * hh + 4;
#pragma unroll
    for (int c = 0; c < 4; ++c) cs2[c] = ldg_nc_v4(t16 + c);
  }
  uint4 cs2[4];
  // valid: the row exists (both lanes of the row agree); w: the half's 64 weights
  __device__ __forceinline__ void finish(uint8_t* tile, int row, int hh, const float* w, float eps, bool valid) const {
    uint8_t* half = tile + hh * kHalfBytes;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(half + sw128_off(row, c));
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = lo16<F16>(u[e]), hi = hi16<F16>(u[e]);
        a0 = fmaf(lo, lo, a0);
        a1 = fmaf(hi, hi, a1);
      }
    }
    float ss = a0 + a1;
    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
    if (!valid) return;
    const float r = rsqrtf(ss * (1.0f / kD) + eps);
    const float4* w4 = reinterpret_cast<const float4*>(w + 64 * hh);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4* p16 = reinterpret_cast<uint4*>(half + sw128_off(row, c));
      const uint4 v = *p16;
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      const uint4 tc = c < 4 ? cs[c] : cs2[c - 4];
      const uint32_t t[4] = {tc.x, tc.y, tc.z, tc.w};
      const float4 wa = w4[2 * c], wb = w4[2 * c + 1];
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      uint32_t out[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&t[e]));  // (cos, sin)
        const float n0 = lo16<F16>(u[e]) * wv[2 * e] * r, n1 = hi16<F16>(u[e]) * wv[2 * e + 1] * r;
        out[e] = pack16<F16>(n0 * sc.x - n1 * sc.y, n0 * sc.y + n1 * sc.x);
      }
      *p16 = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
};

// Prologue of a raw row (bf16 or fp32) read from global memory, used when q/k
// are fp32 (no in-place TMA staging): four lanes per row, lane `quarter`
// (0..3) handling head dims [32 quarter, +32) (chunks 4 quarter .. + 3). Each
// lane sums its squares in order; the row's sum is ((s0 + s1) + (s2 + s3)) by
// two shuffles, so every lane of the warp calls it (valid: the row exists; the
// four lanes of a row agree; an invalid row is written as zeros). Then
// n = x w r and the pair rotation with the fp32 table, rounded once.
template <bool F16>
__device__ __forceinline__ void rope_norm_global_quad(const void* base, int64_t off, int dt,
                                                      const float* __restrict__ w, float eps,
                                                      const float2* __restrict__ tab, uint8_t* tile, int row,
                                                      int quarter, bool valid, uint32_t half) {
  float x[4][8];
  float ss = 0.f;
  if (valid) {
#pragma unroll
    for (int i = 0; i < 4; ++i) load_chunk8(base, off, dt, 4 * quarter + i, x[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[i][e], x[i][e], ss);
    }
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  const float r = rsqrtf(ss * (1.0f / kD) + eps);
  const float4* t4 = reinterpret_cast<const float4*>(tab);
  const float4* w4 = reinterpret_cast<const float4*>(w);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = 4 * quarter + i;
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    if (valid) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float4 cs = __ldg(t4 + 2 * c + hh);
        const float4 ww = __ldg(w4 + 2 * c + hh);
        const float n0 = x[i][4 * hh] * ww.x * r, n1 = x[i][4 * hh + 1] * ww.y * r;
        const float n2 = x[i][4 * hh + 2] * ww.z * r, n3 = x[i][4 * hh + 3] * ww.w * r;
        packed[2 * hh] = pack16<F16>(n0 * cs.x - n1 * cs.y, n0 * cs.y + n1 * cs.x);
        packed[2 * hh + 1] = pack16<F16>(n2 * cs.z - n3 * cs.w, n2 * cs.w + n3 * cs.z);
      }
    }
    *reinterpret_cast<uint4*>(tile + (c >> 3) * half + sw128_off(row, c & 7)) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

}  // namespace st
